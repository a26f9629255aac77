"""Benchmark of the SageAttention3-style attention forward on GB300.

One step = one pass of the whole hot path over one batch of the LLM-prefill
workload (B=2, H=16, L=4096, d=128, non-causal; K carries a per-channel bias):
  sa_quantize (smooth-K mean + NVFP4 quantisation of Q, K, V)
  -> sa_attn_fwd NVFP4 (block-scaled FP4 tcgen05 MMAs, two-level P quantisation)
  -> sa_attn_fwd BF16 (the exact path).
`value` is the NVFP4 path's throughput, 4*B*H*L^2*d / (quantise + fused attention
time), in TOPS, with inputs resident in HBM; the L2 is flushed (a 256 MB write,
then a 256 MB read) before every timed call.  `e2e` is the same metric through the C-ABI call that takes
host buffers, sa_attn_fwd_host: pinned host Q, K, V in, pinned host O out, with
every host <-> device copy inside the timed region (the library overlaps the
copies of one chunk of (batch, kv head) pairs with the compute of the next).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torch.distributed.run (one rank per GPU): the one
problem is sharded by (batch, kv head) pairs -- each rank computes a
contiguous range of pairs with all their query heads (shard.shard_qkv), which
needs no exchange on the data path -- and `value` is the whole problem's
counted work over the max-over-ranks time (strong scaling).
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

WORKLOAD = "llm_prefill"
METRIC = "attention fwd TOPS (4BHL^2d/time), NVFP4 and BF16 paths, 1 GB300; % of peak"
NVFP4_OVER_BF16 = 6.0      # nominal dense FP4 : BF16 tensor ratio on GB300 (13.5 / 2.25 PFLOP/s), for context
# Dense NVFP4 rate measured on this GPU by tests/native/fp4_mma_rate.cu (the
# block-scaled FP4 MMA, M128 x N128|N256 x K64, operands in shared memory):
# FLOP per clock per SM; the FP4 roofline peak is this x SMs x max SM clock.
NVFP4_FLOP_PER_CLK_SM = 32768
# Oracle samples: the cpu_baseline (about 10-20 s of single-threaded NumPy) and
# one step of the reference arm (about 0.2 s: quantising one head dominates).
CPU_SAMPLE_HEADS, CPU_SAMPLE_ROWS = 16, 2048
REF_STEP_ROWS = 16


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sus=p.get("bf16_tflops_sustained"),
                    sm_max_mhz=p.get("sm_max_mhz", 2070.0), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, sm_max_mhz=2070.0, src="fallback")


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
        time.sleep(0.2)
        return self

    def __exit__(self, *a):
        if self.p:
            self.p.terminate()
            self.p.wait()

    def summary(self):
        self.f.seek(0)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            c = [x.strip() for x in line.split(",")]
            if len(c) < 9:
                continue
            try:
                sm.append(float(c[1]))
                mx = float(c[2])
            except ValueError:
                continue
            for n, v in zip(names, c[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_oracle_sample(w, heads, nrows, seed=0):
    """Times the oracle (NVFP4 quantiser + tile-by-tile SA3 emulation, as it
    stands) on `heads` heads x `nrows` query rows of the workload; returns
    (seconds, counted flops of the sampled rows, description)."""
    import numpy as np
    from oracle import attention as A
    x = W.make_inputs(w)
    Lq, L = W.lq(w), w["L"]
    rows = np.array(W.sample_rows(Lq, nrows, seed=seed))
    G = w["H"] // w["Hkv"]
    t0 = time.perf_counter()
    for h in range(heads):
        q = x["q"][0:1, h:h + 1].float().numpy()
        k = x["k"][0:1, h // G:h // G + 1].float().numpy()
        v = x["v"][0:1, h // G:h // G + 1].float().numpy()
        (qd, kd, vd), _ = A.dequantized_operands(q, k, v)
        A.sa3_emulated_attention(qd, kd, vd, w["causal"], rows=rows)
    dt = time.perf_counter() - t0
    if w["causal"] and Lq == L:
        fl = 4.0 * heads * len(rows) * L * w["d"] / 2          # the halved count of the metric
    elif w["causal"]:
        fl = 4.0 * heads * w["d"] * sum(int(r) + L - Lq + 1 for r in rows)
    else:
        fl = 4.0 * heads * len(rows) * L * w["d"]
    desc = (f"{heads} head(s) x {len(rows)} query rows of {w['name']} (full-length keys): NumPy oracle "
            "quantiser (K mean, Q/K/V NVFP4) + SA3 tile-by-tile emulation")
    return dt, fl, desc


def workload_str(w):
    lens = f"L={w['L']}" if W.lq(w) == w["L"] else f"Lq={W.lq(w)} Lkv={w['L']}"
    return f"{w['name']}: B={w['B']} H={w['H']} Hkv={w['Hkv']} {lens} d={w['d']}"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = W.spec(args.workload)
    vals = []
    for i in range(args.warmup + args.steps):
        dt, fl, desc = cpu_oracle_sample(w, heads=1, nrows=REF_STEP_ROWS, seed=i)
        if i >= args.warmup:
            vals.append(fl / dt / 1e12)
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": "f64/f32 (CPU oracle)", "data": "synthetic",
            "config": {"workload": f"{workload_str(w)} {'causal' if w['causal'] else 'non-causal'}",
                       "sample": desc},
            "cpu_baseline": {"value": v, "unit": "TOPS", "cores": host_cores(), "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import quantized_attention_x16_gb300 as sa
    from quantized_attention_x16_gb300 import shard

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = W.spec(args.workload)
    B, H, Hkv, L, d = w["B"], w["H"], w["Hkv"], w["L"], w["d"]
    Lq = W.lq(w)                                   # query rows (L: keys)
    x = W.make_inputs(w)
    fl = W.flops(w)                                # the whole problem's counted work
    causal = w["causal"]
    # this rank's share: a contiguous range of (batch, kv head) pairs with all
    # their query heads, as a problem of its own (B = 1, H = n*G, Hkv = n)
    p0, p1 = shard.pair_range(B, Hkv, world, rank)
    if world > 1:
        qs, ks, vs = shard.shard_qkv(x["q"], x["k"], x["v"], world, rank)
        x = dict(q=qs.contiguous(), k=ks.contiguous(), v=vs.contiguous())
        B, H, Hkv = 1, (p1 - p0) * (H // Hkv), p1 - p0
    if p1 == p0:
        raise SystemExit(f"rank {rank}: no (batch, kv head) pair to compute ({w['B'] * w['Hkv']} pairs, {world} ranks)")
    q, k, v = (x[n].to(dev) for n in "qkv")
    # A one-token query (decode) against a GQA cache: the G query heads of a
    # kv head read the same keys and values, and with one row per head no mask
    # tells them apart (under the bottom-right causal mask the row sees every
    # key), so Q [B, H, 1, d] goes to the library as [B, Hkv, G, d] -- the
    # same BHLD memory, G query rows per kv head, the same O -- with G times
    # fewer 128-row query tiles.
    fold = Lq == 1 and H > Hkv
    if fold:
        q, H, Lq, causal = q.view(B, Hkv, H // Hkv, d), Hkv, H // Hkv, False
    # at most 16 query rows per kv head: the library's decode kernel (4, 8 or
    # 16 rows), HBM-bound by design; else the prefill kernel
    nr = (H // Hkv) * Lq
    decode = nr <= 16
    kname4 = (f"attn_decode_kernel<{d}, {4 if nr <= 4 else 8 if nr <= 8 else 16}>" if decode
              else f"attn_nvfp4_kernel<{d}>")
    fq = sa.FP4QKV(B, H, Hkv, Lq, d, device=dev, Lkv=L)
    o4 = torch.empty_like(q)
    o16 = torch.empty_like(q)
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    flush_sink = torch.zeros(1, dtype=torch.int64, device=dev)

    def flush_l2():
        # write 256 MB (evicts every line the last step left in the 129 MB L2),
        # then read it back: the write's own dirty lines are written back here,
        # before the timed calls, instead of inside them
        flush.zero_()
        flush_sink.add_(flush.view(torch.int64).sum())

    # the library's work split (stream-K for the NVFP4 path once the pairs
    # fill the SMs, split-KV for problems too small to); the workspace is
    # allocated once, outside the timed region
    ws4 = sa.sa_attn_fwd_workspace_bytes(B, H, Hkv, Lq, d, causal, "nvfp4", 0, Lkv=L)
    ws16 = sa.sa_attn_fwd_workspace_bytes(B, H, Hkv, Lq, d, causal, "bf16", 0, Lkv=L)
    nsplit_ws = max(ws4, ws16)
    ws = torch.empty(max(nsplit_ws, 16), dtype=torch.uint8, device=dev)

    def step(ev):
        # each call timed alone (the breakdown), and the BF16 path
        ev[0].record()
        sa.sa_quantize(q, k, v, out=fq)
        ev[1].record()
        sa.sa_attn_fwd(fq, o=o4, causal=causal, mode="nvfp4", nsplit=0, workspace=ws)
        ev[2].record()
        sa.sa_attn_fwd(q, k, v, o=o16, causal=causal, mode="bf16", nsplit=0, workspace=ws)
        ev[3].record()

    def step_path(ev):
        # the headline path, sa_quantize then the NVFP4 sa_attn_fwd back to
        # back in one interval: the attention launch may overlap the
        # quantiser's last CTAs (programmatic dependent launch), which an
        # event recorded between them would prevent
        ev[0].record()
        sa.sa_quantize(q, k, v, out=fq)
        sa.sa_attn_fwd(fq, o=o4, causal=causal, mode="nvfp4", nsplit=0, workspace=ws)
        ev[1].record()

    # the fused-Q mode (Q quantised inside the attention kernel): K and V
    # through sa_quantize_kv, bf16 Q straight into the attention kernel; the
    # same work and the same O bytes as the path above (prefill shapes only)
    fk = None if decode else sa.FP4QKV(B, H, Hkv, Lq, d, device=dev, Lkv=L)

    def step_fq(ev):
        # ev[0..2]: the two calls timed apart; ev[3..4]: back to back, after
        # another L2 flush
        ev[0].record()
        sa.sa_quantize_kv(k, v, H, Lq=Lq, out=fk)
        ev[1].record()
        sa.sa_attn_fwd(q, fk, o=o4, causal=causal, mode="nvfp4_fq", nsplit=0, workspace=ws)
        ev[2].record()
        flush_l2()
        ev[3].record()
        sa.sa_quantize_kv(k, v, H, Lq=Lq, out=fk)
        sa.sa_attn_fwd(q, fk, o=o4, causal=causal, mode="nvfp4_fq", nsplit=0, workspace=ws)
        ev[4].record()

    for _ in range(args.warmup):
        flush_l2()
        step([torch.cuda.Event(enable_timing=True) for _ in range(4)])
        flush_l2()
        step_path([torch.cuda.Event(enable_timing=True) for _ in range(2)])
        if fk is not None:
            flush_l2()
            step_fq([torch.cuda.Event(enable_timing=True) for _ in range(5)])
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == sa.SA_OK

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    evf = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(local_rank) as clk:
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush_l2()
            step(evs[i])
            flush_l2()
            step_path(evp[i])
            if fk is not None:
                flush_l2()
                step_fq(evf[i])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    # sa_quantize: 2 kernels; each attention call: 1, plus a combine kernel
    # when its work is split; per step the breakdown and the path
    n4 = 2 if ws4 > 0 else 1
    launches = args.steps * ((2 + n4 + (2 if ws16 > 0 else 1)) + (2 + n4) + (2 * (2 + n4) if fk is not None else 0))
    tq = [a[0].elapsed_time(a[1]) * 1e-3 for a in evs]
    t4 = [a[1].elapsed_time(a[2]) * 1e-3 for a in evs]
    t16 = [a[2].elapsed_time(a[3]) * 1e-3 for a in evs]
    tp = [a[0].elapsed_time(a[1]) * 1e-3 for a in evp]
    mean = lambda xs: sum(xs) / len(xs)   # noqa: E731
    t_q, t_4, t_16, t_path = mean(tq), mean(t4), mean(t16), mean(tp)
    fq_times = None
    if fk is not None:
        fq_times = {"quantize_kv_us": mean([a[0].elapsed_time(a[1]) for a in evf]) * 1e3,
                    "attn_us": mean([a[1].elapsed_time(a[2]) for a in evf]) * 1e3,
                    "path_us": mean([a[3].elapsed_time(a[4]) for a in evf]) * 1e3}
    # rank 0's own launches for the per-kernel rooflines (its share of the problem)
    # (a folded decode: H = Hkv heads of Lq = G rows each, the same work)
    w_local = dict(w, B=B, H=H, Hkv=Hkv, Lq=Lq, causal=causal)
    fl_local = W.flops(w_local)
    lq_, l4_, l16_ = t_q, t_4, t_16
    # the slowest rank sets each time of the whole problem (no-ops at N = 1)
    t_path, t_q, t_4, t_16 = (shard.max_over_ranks(t, device=dev) for t in (t_path, t_q, t_4, t_16))
    assert sa.sa_last_device_error() == sa.SA_OK

    # ---- end to end through the public API with host buffers (same metric)
    # sa_attn_fwd_host: pinned host Q, K, V in, pinned host O out; the library
    # chunks the problem by (batch, kv head) and overlaps its copies with the
    # quantiser and attention kernels of neighbouring chunks.  It takes one
    # length for queries and keys, so a workload with Lq != L has no e2e.
    e2e = None
    if Lq == L:
        hq, hk, hv = (x[n].pin_memory() for n in "qkv")
        ho = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
        d2h = ho.numel() * ho.element_size()
        ws = torch.empty(sa.sa_attn_fwd_host_workspace_bytes(B, H, Hkv, L, d, "nvfp4"), dtype=torch.uint8,
                         device=dev)
        del fq

        # SA_HOST_OVERLAP: each step's inputs are final when it is called, so
        # its first copies may run beside the previous step's last compute and
        # copy-out (every step still copies its own inputs in and its O out)
        def e2e_step():
            sa.sa_attn_fwd_host(hq, hk, hv, o=ho, causal=causal, mode="nvfp4", workspace=ws, overlap=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            e2e_step()
        e1.record()
        torch.cuda.synchronize()
        t_e2e = shard.max_over_ranks(e0.elapsed_time(e1) * 1e-3 / args.steps, device=dev)
        e2e = {"value": fl / t_e2e / 1e12, "unit": "TOPS", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3,
               "api": "sa_attn_fwd_host (nvfp4, SA_HOST_OVERLAP)"}

    if rank != 0:
        return
    pk = peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    nvfp4_peak = NVFP4_FLOP_PER_CLK_SM * sms * pk["sm_max_mhz"] * 1e6 / 1e12
    nvfp4_nominal_ratio_peak = pk["bf16"] * NVFP4_OVER_BF16
    a4 = fl_local / l4_ / 1e12                     # rank 0's launch: its share over its own time
    a16 = fl_local / l16_ / 1e12
    qbytes = quant_bytes(w_local)
    attn_bytes = attn_nvfp4_bytes(w_local)
    clocks = clk.summary()
    prof = load_profile_traffic()
    cpu = None
    if not args.skip_cpu_baseline:
        cpu_dt, cpu_fl, cpu_desc = cpu_oracle_sample(w, heads=CPU_SAMPLE_HEADS, nrows=CPU_SAMPLE_ROWS)
        cpu = {"value": cpu_fl / cpu_dt / 1e12, "unit": "TOPS", "cores": host_cores(), "kind": "oracle",
               "sample": cpu_desc, "seconds": cpu_dt}
    line = {
        "metric": METRIC,
        "value": fl / t_path / 1e12,
        "unit": "TOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_path * 1e3,
        "higher_is_better": True,
        "scaling": "strong",
        "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x e4m3-scaled, fp32 accumulate); bf16 path alongside",
        "data": "synthetic (seeded torch.Generator, bf16)",
        "config": {"workload": f"{workload_str(w)} {'causal' if causal else 'non-causal'} ({w['kind']} inputs)",
                   "B": w["B"], "H": w["H"], "Hkv": w["Hkv"], "L": L, "Lq": W.lq(w), "d": d, "causal": w["causal"],
                   "gqa_fold": ("Q [B, H, 1, d] passed as [B, Hkv, H/Hkv, d]: the query heads of a kv head as "
                                "its query rows") if fold else None,
                   "l2": "flushed before every timed call by a 256 MB write and a 256 MB read",
                   "value_def": "4*B*H*L^2*d of the whole problem (halved for causal; with Lq != L, 4*B*H*d x "
                                "the (query, key) pairs the mask leaves) / the slowest rank's (sa_quantize + "
                                "NVFP4 sa_attn_fwd, back to back in one CUDA-event interval)",
                   "parallelism": (f"(batch, kv head) pairs sharded over {world} GPUs, {p1 - p0} of "
                                   f"{w['B'] * w['Hkv']} on rank 0, no collective on the data path")
                                  if world > 1 else "one GPU, the whole problem",
                   "work_split": "library choice (sa_attn_fwd_ws, nsplit=0): nvfp4 "
                                 + ("stream-K/split" if ws4 > 0 else "one unit per CTA") + ", bf16 "
                                 + ("split-KV" if ws16 > 0 else "one unit per CTA")},
        "paths": {
            "nvfp4_attn_only_tops": a4,
            "nvfp4_attn_us": t_4 * 1e6,
            "quantize_us": t_q * 1e6,
            "quantize_gbs": qbytes / lq_ / 1e9,
            "path_us": t_path * 1e6,
            "quantize_plus_attn_timed_apart_us": (t_q + t_4) * 1e6,
            "nvfp4_end_to_end_tops": fl / t_path / 1e12,
            "bf16_tflops": a16,
            "bf16_attn_us": t_16 * 1e6,
            "bf16_frac_of_measured_peak": a16 / pk["bf16"],
            "fused_q": (dict(fq_times, attn_traffic_bytes=prof.get("attn_nvfp4_fq"), note="mode nvfp4_fq: sa_quantize_kv + the attention kernel quantising "
                             "bf16 Q itself (bit-identical O); path_us against path_us above, L2 flushed before "
                             "each interval") if fq_times is not None else None),
        },
        "roofline": {"kernel": kname4, "bound": "tensor", "achieved": a4, "peak": nvfp4_peak,
                     "unit": "TFLOP/s", "frac": a4 / nvfp4_peak,
                     "traffic": prof.get("attn_decode" if decode else "attn_nvfp4"),
                     "peak_src": (f"measured NVFP4 MMA rate {NVFP4_FLOP_PER_CLK_SM} FLOP/clk/SM (fp4_mma_rate probe) x {sms} "
                                  f"SMs x {pk['sm_max_mhz']} MHz max SM clock"),
                     "peak_nominal_ratio": nvfp4_nominal_ratio_peak,
                     "frac_of_nominal_ratio_peak": a4 / nvfp4_nominal_ratio_peak,
                     "peak_nominal_ratio_src": f"{pk['src']} bf16 burst {pk['bf16']} x nominal FP4:BF16 ratio "
                                               f"{NVFP4_OVER_BF16}"},
        "roofline_secondary": mufu_roofline(a4, d, pk),
        "roofline_bf16": {"kernel": f"attn_bf16_kernel<{d}>", "bound": "tensor", "achieved": a16, "peak": pk["bf16"],
                          "unit": "TFLOP/s", "frac": a16 / pk["bf16"], "traffic": prof.get("attn_bf16"),
                          "peak_src": f"{pk['src']} bf16 burst"},
        "roofline_quantize": {"kernel": f"sa_quantize (quant_kernel<{d}, 1> + quant_kernel<{d}, 2>)", "bound": "hbm",
                              "achieved": qbytes / lq_ / 1e9,
                              "peak": pk["hbm"], "unit": "GB/s", "frac": qbytes / lq_ / 1e9 / pk["hbm"],
                              "traffic": (prof["quant_pass1"] + prof["quant_pass2"]
                                          if "quant_pass1" in prof and "quant_pass2" in prof else None),
                              "algorithmic_bytes": qbytes,
                              "traffic_kernels": {"pass 1 (Q, K mean)": prof.get("quant_pass1"),
                                                  "pass 2 (V, K')": prof.get("quant_pass2")}},
        "roofline_hbm_attn": {"kernel": kname4, "bound": "hbm" + ("" if decode else " (context: the bound of "
                              "few-query shapes such as decode)"), "achieved": attn_bytes / l4_ / 1e9,
                              "peak": pk["hbm"], "unit": "GB/s", "frac": attn_bytes / l4_ / 1e9 / pk["hbm"],
                              "traffic": prof.get("attn_decode") if decode else None,
                              "algorithmic_bytes": attn_bytes},
        "cpu_baseline": cpu,
        "e2e": e2e if e2e is not None else {"value": None, "unit": "TOPS", "h2d_bytes_per_step": 0,
                                            "d2h_bytes_per_step": 0,
                                            "note": "sa_attn_fwd_host takes equal query and key lengths"},
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if decode:
        # the decode kernel reads the whole K/V cache once per call: its
        # primary roofline is HBM; the tensor figure stays beside it
        line["roofline_tensor"] = line["roofline"]
        line["roofline"] = line.pop("roofline_hbm_attn")
    print(json.dumps(line), flush=True)


# Exponentials per SM per clock on this GPU (ex2.approx: measured with a
# throughput probe of independent chains over the whole device).
MUFU_EX2_PER_SM_CLK = 32


def mufu_roofline(achieved_tops, d, pk):
    """Secondary bound of the fused attention: one ex2 per score element on the
    MUFU, 4*d flops per element, at the maximum SM clock."""
    try:
        import torch
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    except Exception:
        sms = 152
    peak = MUFU_EX2_PER_SM_CLK * 4 * d * sms * pk["sm_max_mhz"] * 1e6 / 1e12
    return {"kernel": f"attn_nvfp4_kernel<{d}>", "bound": "alu (MUFU ex2, one per score)", "achieved": achieved_tops,
            "peak": peak, "unit": "TOPS", "frac": achieved_tops / peak,
            "peak_src": f"{MUFU_EX2_PER_SM_CLK} ex2/clk/SM (measured) x 4d flops x {sms} SMs x {pk['sm_max_mhz']} MHz"}


def quant_bytes(w):
    """Algorithmic HBM bytes of sa_quantize: read Q, K, V (bf16) + K again for the
    mean, write codes (0.5 B/elem) and scales (1/16 B/elem), the mean and its partials."""
    B, H, Hkv, L, d = w["B"], w["H"], w["Hkv"], w["L"], w["d"]
    nq, nk = B * H * W.lq(w) * d, B * Hkv * L * d
    reads = 2 * nq + 2 * nk * 2 + 2 * nk
    writes = (nq + 2 * nk) * (0.5 + 1 / 16)
    return reads + writes


def attn_nvfp4_bytes(w):
    """Algorithmic HBM bytes of one NVFP4 attention call: read the FP4 codes and
    e4m3 scales of Q, K, V once (0.5 + 1/16 B per element of the problem, no
    tile padding), write O (bf16)."""
    B, H, Hkv, L, d = w["B"], w["H"], w["Hkv"], w["L"], w["d"]
    Lq = W.lq(w)
    fp4 = 0.5 + 1 / 16
    return (B * H * Lq * d + 2 * B * Hkv * L * d) * fp4 + 2 * B * H * Lq * d


def load_profile_traffic():
    """DRAM bytes per launch recorded from ncu captures (profiles/traffic.json),
    kept only for kernels whose sources still hash to the captured version."""
    import hashlib
    out = {}
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
    except Exception:
        return out
    for name, rec in t.items():
        if not isinstance(rec, dict) or "sources" not in rec:
            continue
        h = hashlib.sha256()
        try:
            for src in rec["sources"]:
                with open(os.path.join(ROOT, "quantized_attention_x16_gb300", "csrc", src), "rb") as f:
                    h.update(f.read())
        except OSError:
            continue
        if h.hexdigest()[:16] == rec.get("sha256_16"):
            out[name] = rec["bytes"]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(W.WORKLOADS),
                    help="another workload (profiling and sweeps; the headline is llm_prefill)")
    ap.add_argument("--skip-cpu-baseline", action="store_true",
                    help="omit the oracle timing (profiling runs)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
