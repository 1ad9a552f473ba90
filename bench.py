"""Benchmark of the TurboQuant hot path on B300: long-context batched decode over a
compressed KV cache.

Workload (one step = one decode step of every sequence):
  batch 8, 8 KV heads, 32 query heads (GQA groups of 4), head_dim 128, 131072 cached tokens
  (bf16 keys/values from the anisotropic generator, quantized at prefill: keys 3 bits =
  2-bit codes + 1 QJL bit, values 3-bit MSE-only codes), then per step:
    append the new token's key and value (rotate + code + pack, QJL signs for the key),
    advance the lengths, score all cached keys (attention logits, written to HBM), then the
    softmax over those logits and the weighted sum of the dequantized values.
Metric: compressed-key logit scores per second (query heads x cached keys / time), plus
the HBM bandwidth those kernels achieve.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tq|reference]
Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a bounded sample.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

B, HKV, G, D, N0 = 8, 8, 4, 128, 131072
HQ = HKV * G
KBITS, VBITS = 3, 3
SEED_ROT, SEED_DATA = 0, 3
METRIC = "compressed-key logit scores/sec and achieved HBM GB/s (% of B300 roofline)"
UNIT = "logit scores/s"
WORKLOAD = ("long-context batched decode: batch 8, 8 KV heads, 32 query heads, head_dim 128, "
            "131072 cached tokens + 1 appended per step; keys 3 bits (2 MSE + 1 QJL), values 3-bit MSE")

# Algorithmic bytes per cached key for one (batch, KV head) group at d = 128
K_BYTES = 2 * 16 + 16 + 2 + 2        # 2 code planes, sign words, norm, residual norm = 52
V_BYTES = 3 * 16 + 2                 # 3 code planes + norm = 50
LOGIT_BYTES = K_BYTES + G * 4        # keys read + 4 fp32 logits written = 68
VALUES_BYTES = G * 4 + V_BYTES       # 4 logits read + value codes read = 66


def set_batch(b: int) -> None:
    global B, WORKLOAD
    if b != B:
        WORKLOAD = WORKLOAD.replace("batch 8", f"batch {b}")
        B = b


# DRAM traffic of the decode kernels from one-kernel ncu captures (dram__bytes_read.sum +
# dram__bytes_write.sum; batch 2 of the same workload, one launch, scaled to a launch here by the
# keys it scores).  A figure is reported only while the sources it was taken on are unchanged.
NCU_CAPTURES = {
    # values_coded128_kernel<3, false>: 138.446 MB read + 2.834 MB written, 2 x 8 x 131071 keys
    "attn_values": (['k_attn.cu', 'attn_q8.cuh', 'lut.cuh', 'values.cuh', 'tq_device.cuh', 'tq_internal.h'], "b83f70a6c3e9b48a", (138.445568e6 + 2.83392e6) / (2 * 8 * 131071)),
    # logits_tc_kernel<2>: 109.181 MB read + 13.929 MB written (part of the logits still in L2)
    "attn_logits": (['k_logits_tc.cu', 'tcgen05.cuh', 'mma_e4m3.cuh', 'k_attn.cu', 'lut.cuh', 'attn_q8.cuh', 'tq_device.cuh', 'tq_internal.h'], "0f385a557dd290bb",
                    (109.18144e6 + 13.929472e6) / (2 * 8 * 131071)),
}


def ncu_traffic(kernel: str, keys: float):
    if kernel not in NCU_CAPTURES:
        return None
    sources, sha, per_key = NCU_CAPTURES[kernel]
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "compressed_kv_cache_02_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if per_key is None or h.hexdigest()[:16] != sha:
        return None
    return per_key * keys


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


def _bf16_peak():
    """Dense bf16 TFLOP/s: the measured burst figure (a kernel timed alone), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        if j.get("bf16_tflops"):
            return float(j["bf16_tflops"]), "measured"
    return 1800.0, "fallback"


BF16_PEAK = _bf16_peak()


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""
    FIELDS = "clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown," \
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 6:
                self.rows.append(parts)

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in self.rows for k in range(4) if r[2 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- the TQ arm

def build_state(dev):
    from compressed_kv_cache_02_b300 import inputs, tq
    kctx = tq.Context(D, KBITS, seed=SEED_ROT)
    vctx = tq.Context(D, VBITS, seed=SEED_ROT + 1, mode=tq.TQ_MODE_MSE)
    cap = N0 + 4096
    kc = kctx.alloc_codes(B, HKV, cap, device=dev)
    vc = vctx.alloc_codes(B, HKV, cap, device=dev)
    kfac = inputs.anisotropic_factors(HKV, D, seed=SEED_DATA, device=dev)
    vfac = inputs.anisotropic_factors(HKV, D, seed=SEED_DATA + 1000, device=dev)
    t_pre = 0.0
    for b in range(B):   # prefill one batch row at a time: 2 x 256 MB of bf16 at a time
        K = inputs.anisotropic(1, HKV, N0, D, kfac, seed=SEED_DATA * 100 + b, device=dev)
        V = inputs.anisotropic(1, HKV, N0, D, vfac, seed=SEED_DATA * 100 + 1000 + b, device=dev)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for h in range(HKV):
            kctx.quantize(K[0, h], out=tq.Codes(kc.planes[b, h, :N0], kc.norm[b, h, :N0], kc.signs[b, h, :N0],
                                                kc.rnorm[b, h, :N0]))
            vctx.quantize(V[0, h], out=tq.Codes(vc.planes[b, h, :N0], vc.norm[b, h, :N0]))
        e1.record()
        torch.cuda.synchronize()
        t_pre += e0.elapsed_time(e1) / 1e3
        del K, V
    flags = kctx.sync_status() | vctx.sync_status()
    if flags:
        raise RuntimeError(f"device error flags {flags} after prefill")
    return dict(kctx=kctx, vctx=vctx, kc=kc, vc=vc, cap=cap, kfac=kfac, vfac=vfac,
                prefill_s=t_pre, prefill_vectors=2 * B * HKV * N0)


def step_inputs(state, nsteps, dev):
    """Per step: the new key and value [B, Hkv, d] (bf16) and the queries [B, Hq, d] (fp32)."""
    from compressed_kv_cache_02_b300 import inputs
    K = inputs.anisotropic(B, HKV, nsteps, D, state["kfac"], seed=10_000, device=dev)
    V = inputs.anisotropic(B, HKV, nsteps, D, state["vfac"], seed=20_000, device=dev)
    Q = inputs.anisotropic(B, HKV, nsteps * G, D, state["kfac"], seed=30_000, device=dev, dtype=torch.float32)
    Q = Q.reshape(B, HKV, nsteps, G, D)
    ks = [K[:, :, s].contiguous() for s in range(nsteps)]
    vs = [V[:, :, s].contiguous() for s in range(nsteps)]
    qs = [Q[:, :, s].reshape(B, HQ, D).contiguous() for s in range(nsteps)]
    return ks, vs, qs


def run_tq(args, world, rank, local):
    from compressed_kv_cache_02_b300 import tq
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    state = build_state(dev)
    kctx, vctx, kc, vc, cap = state["kctx"], state["vctx"], state["kc"], state["vc"], state["cap"]
    paths = {"auto": tq.TQ_PATH_AUTO, "cuda_core": tq.TQ_PATH_CUDA_CORE, "tensor": tq.TQ_PATH_TENSOR}
    kctx.set_kernel_path(paths[args.kernel_path])
    vctx.set_kernel_path(paths[args.values_path or args.kernel_path])
    total = args.warmup + args.steps
    assert N0 - args.warmup >= 1 and N0 + args.steps <= cap
    ks, vs, qs = step_inputs(state, total, dev)
    length = torch.full((B,), N0 - args.warmup, dtype=torch.int32, device=dev)
    logits = torch.empty(B, HQ, cap, device=dev)
    out = torch.empty(B, HQ, D, device=dev)
    ws = kctx.attn_workspace(B, HQ, HKV, cap, device=dev)
    scale = 1.0 / D ** 0.5
    stream = torch.cuda.current_stream()

    vws = tq.values_workspace(D, B, HQ, HKV, cap, device=dev)
    # The value append runs on a side stream, overlapped with the key append and the logits: it
    # writes at the step's old lengths (a copy taken first, as advance_len changes `length`), and
    # only the value sum waits for it.
    side = torch.cuda.Stream(device=dev)
    pos = torch.empty_like(length)
    forked, joined = torch.cuda.Event(), torch.cuda.Event()

    def step_calls(k, v, q):
        pos.copy_(length)
        forked.record(stream)
        side.wait_event(forked)
        vctx.append(v, vc, cap, pos, stream=side)
        joined.record(side)
        kctx.append(k, kc, cap, pos)
        kctx.advance_len(length, cap)
        yield
        kctx.attn_logits(q, kc, cap, length, scale, out=logits, workspace=ws)
        yield
        stream.wait_event(joined)
        tq.attn_values(logits, length, vc, vctx=vctx, out=out, workspace=vws)

    def step(s, ev=None):
        if ev:
            ev[3].record()
        calls = step_calls(ks[s], vs[s], qs[s])
        next(calls)
        if ev:
            ev[0].record()
        next(calls)
        if ev:
            ev[1].record()
        next(calls, None)
        if ev:
            ev[2].record()

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    if kctx.sync_status() or vctx.sync_status():
        raise RuntimeError("device error flags after warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    lens_timed = [N0 + s + 1 for s in range(args.steps)]    # cache length seen by step s
    barrier(world)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        t0.record(stream)
        for s in range(args.steps):
            step(args.warmup + s, evs[s])
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed = max_over_ranks(t0.elapsed_time(t1) / 1e3, world)
    if kctx.sync_status() or vctx.sync_status():
        raise RuntimeError("device error flags after the timed steps")
    t_logits = [e[0].elapsed_time(e[1]) / 1e3 for e in evs]
    t_output = [e[1].elapsed_time(e[2]) / 1e3 for e in evs]
    t_append = [e[3].elapsed_time(e[0]) / 1e3 for e in evs]
    keys = sum(lens_timed) * B * HKV
    scores = keys * G
    value = scores * world / elapsed

    # end to end through the public API: pinned host inputs in, the step's output back out
    hk = [k.cpu().pin_memory() for k in ks]
    hv = [v.cpu().pin_memory() for v in vs]
    hq = [q.cpu().pin_memory() for q in qs]
    hout = torch.empty(B, HQ, D).pin_memory()
    dk, dv, dq = torch.empty_like(ks[0]), torch.empty_like(vs[0]), torch.empty_like(qs[0])
    length.fill_(N0 - args.warmup)
    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(args.steps):
        i = args.warmup + s
        dk.copy_(hk[i], non_blocking=True)
        dv.copy_(hv[i], non_blocking=True)
        dq.copy_(hq[i], non_blocking=True)
        for _ in step_calls(dk, dv, dq):
            pass
        hout.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_elapsed = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    h2d = dk.numel() * dk.element_size() + dv.numel() * dv.element_size() + dq.numel() * 4
    d2h = hout.numel() * 4

    hbm, peak_kind = peaks()
    logits_bytes = [LOGIT_BYTES * B * HKV * L for L in lens_timed]
    output_bytes = [VALUES_BYTES * B * HKV * L for L in lens_timed]
    gbs_logits = sum(logits_bytes) / sum(t_logits) / 1e9
    gbs_output = sum(output_bytes) / sum(t_output) / 1e9
    dominant = "attn_values" if sum(t_output) >= sum(t_logits) else "attn_logits"
    dom_gbs = gbs_output if dominant == "attn_values" else gbs_logits
    launches_per_step = 3 + 3 + 2   # append x2 + advance; logits: prep x2 + kernel; values: partial + combine
    step_bytes = (sum(logits_bytes) + sum(output_bytes)) / args.steps
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": B, "kv_heads": HKV, "query_heads": HQ, "head_dim": D,
                   "cached_tokens": N0, "key_bits": KBITS, "value_bits": VBITS, "parallelism": f"replicas x{world}",
                   "kernel_path": args.kernel_path, "values_path": args.values_path or args.kernel_path,
                   "l2": "inputs larger than L2 (cache codes ~0.9 GB)"},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": dom_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": dom_gbs / hbm, "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": (ncu_traffic(dominant, statistics.mean(lens_timed) * B * HKV)
                                 if args.kernel_path == "auto" else None),
                     "traffic_unit": "bytes per launch (ncu, scaled from batch 2)"},
        "kernels": {
            "attn_logits": {"ms": statistics.mean(t_logits) * 1e3, "GB_s": gbs_logits,
                            "bytes_per_key": LOGIT_BYTES, "frac_of_measured": gbs_logits / hbm,
                            "frac_of_8TBs": gbs_logits / 8000.0},
            "attn_values": {"ms": statistics.mean(t_output) * 1e3, "GB_s": gbs_output,
                            "bytes_per_key": VALUES_BYTES, "frac_of_measured": gbs_output / hbm,
                            "frac_of_8TBs": gbs_output / 8000.0},
            "append_K_V_and_advance": {"ms": statistics.mean(t_append) * 1e3,
                                       "note": "key append + advance on the main stream; the value append "
                                               "overlaps them and the logits on a side stream"},
            "step_GB_s": step_bytes / (elapsed / args.steps) / 1e9,
            "prefill_quantize": {"vectors": state["prefill_vectors"], "s": state["prefill_s"],
                                 "vectors_per_s": state["prefill_vectors"] / state["prefill_s"]},
        },
        "e2e": {"value": scores * world / e2e_elapsed, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu:
        res["cpu_baseline"] = cpu_baseline(args, budget_s=args.cpu_seconds)
    if not args.no_extra:
        del logits, ws, vws, kc, vc
        paged = measure_paged(dev, state=state)   # the same prefilled cache, moved into pages
        del state
        torch.cuda.empty_cache()
        res["other_workloads"] = {"search": measure_search(dev), "prefill": measure_prefill(dev),
                                  "fractional": measure_fractional(dev), "decode1": measure_decode1(dev),
                                  "paged": paged, "polar": measure_polar(dev)}
    return res


# ----------------------------------------------------------------------------- secondary workloads

def _event_time(fn, reps=1):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        out = fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps, out


def measure_search(dev):
    """Vector search: 10^6 unit vectors (d=200, cone law) coded at 2 and 4 total bits, 10^4
    queries, top-100 (top-1 and top-10 are its prefixes); recall@1@k against the exact fp32
    top-1 (fp32 GEMM, TF32 off)."""
    from compressed_kv_cache_02_b300 import inputs, tq
    d, n, nq, k = 200, 1_000_000, 10_000, 100
    X = inputs.cone(n, d, seed=5, mu_seed=55, device=dev)
    Q = inputs.cone(nq, d, seed=6, mu_seed=55, device=dev)
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    true1 = torch.cat([torch.argmax(Q[i:i + 1000] @ X.T, dim=1) for i in range(0, nq, 1000)])
    torch.backends.cuda.matmul.allow_tf32 = prev
    res = {}
    for bits in (2, 4):
        ctx = tq.Context(d, bits, seed=0)
        db = ctx.alloc_codes(n, device=dev)
        ctx.quantize(X, out=db)
        t_index, _ = _event_time(lambda: ctx.quantize(X, out=db))
        ws = ctx.search_workspace(nq, n, k, device=dev)
        ctx.search_topk(Q, db, k, workspace=ws)
        t_search, (sc, idx) = _event_time(lambda: ctx.search_topk(Q, db, k, workspace=ws))
        hit = idx.long() == true1[:, None]
        recall = {f"recall@1@{kk}": float(hit[:, :kk].any(dim=1).float().mean()) for kk in (1, 10, 100)}
        code_bytes = (ctx.P * ctx.W + ctx.Ws) * 4 + 4
        res[f"{bits}bit"] = {"search_ms": t_search * 1e3, "pairs_per_s": n * nq / t_search,
                             "index_ms": t_index * 1e3, "index_vectors_per_s": n / t_index,
                             "db_bytes_per_vector": code_bytes, **recall}
        del db, ws
    return {"workload": "1e6 cone vectors d=200, 1e4 queries, top-100", **res}


def _decode_codes(ctx, codes, Pi, cent):
    """x_hat = n16 Pi^T c[idx] from packed codes, in torch (measurement only)."""
    planes = codes.planes.view(torch.int32)
    n, P, W = planes.shape
    j = torch.arange(ctx.d, device=planes.device)
    idx = torch.zeros(n, ctx.d, dtype=torch.long, device=planes.device)
    for p in range(P):
        words = planes[:, p, :].long() & 0xFFFFFFFF
        idx |= ((words[:, j // 32] >> (j % 32)) & 1) << p
    nrm = codes.norm.view(torch.float16).float()
    return nrm[:, None] * (cent[idx] @ Pi)


def measure_prefill(dev):
    """Prefill-time bulk quantization: 32 layers x 8 KV heads x 16384 tokens x d=128 (bf16,
    anisotropic), MSE bits 2, 3, 4 plus 1 QJL bit.  Throughput of the quantize kernel and the
    distortions D_mse = E||x - x_hat||^2/||x||^2 (2^16 sampled vectors) and D_prod =
    E(est - <q,x>)^2 / (||q||^2 ||x||^2) (1024 queries x 2^14 sampled keys, est from the logits
    kernel with scale 1)."""
    from compressed_kv_cache_02_b300 import inputs, tq
    L_, H_, T_ = 32, 8, 16384
    n = L_ * H_ * T_
    fac = inputs.anisotropic_factors(H_, D, seed=4, device=dev)
    X = inputs.anisotropic(L_, H_, T_, D, fac, seed=4, device=dev).reshape(n, D)
    Qs = inputs.anisotropic(1, 1, 1024, D, (fac[0][:1], fac[1][:1]), seed=40, device=dev,
                            dtype=torch.float32).reshape(1024, D)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    sample = torch.randperm(n, generator=g, device=dev)[: 1 << 16]
    res = {}
    for bits in (3, 4, 5):
        ctx = tq.Context(D, bits, seed=0)
        out = ctx.alloc_codes(n, device=dev)
        ctx.quantize(X, out=out)
        t, _ = _event_time(lambda: ctx.quantize(X, out=out))
        Pi, _, cent, _ = ctx.export()
        Pi_t = torch.from_numpy(Pi).to(dev)
        cent_t = torch.from_numpy(cent).float().to(dev)
        xs = X[sample].float()
        sub = tq.Codes(out.planes[sample], out.norm[sample], out.signs[sample], out.rnorm[sample])
        xh = _decode_codes(ctx, sub, Pi_t, cent_t)
        d_mse = float(((xs - xh) ** 2).sum(1).div(xs.pow(2).sum(1)).mean())
        ks = 1 << 14
        keys = tq.Codes(sub.planes[:ks].reshape(1, 1, ks, ctx.P, -1), sub.norm[:ks].reshape(1, 1, ks),
                        sub.signs[:ks].reshape(1, 1, ks, -1), sub.rnorm[:ks].reshape(1, 1, ks))
        est = ctx.attn_logits(Qs.reshape(1, 1024, D), keys, ks, torch.tensor([ks], dtype=torch.int32, device=dev),
                              1.0)[0]
        exact = Qs @ xs[:ks].T
        den = Qs.pow(2).sum(1)[:, None] * xs[:ks].pow(2).sum(1)[None, :]
        d_prod = float(((est - exact) ** 2 / den).mean())
        bytes_per_vec = 2 * D + (ctx.P * ctx.W + ctx.Ws) * 4 + 4
        # the rotation and the JL projection: 2 d (d + m) algorithmic flops per vector (the bf16
        # pieces the kernel splits its operands into are not counted)
        tflops = 2 * D * (D + ctx.m) * n / t / 1e12
        res[f"{bits - 1}+1bit"] = {"quantize_ms": t * 1e3, "vectors_per_s": n / t,
                                  "GB_s": n * bytes_per_vec / t / 1e9, "GB_s_frac_of_measured_hbm": None,
                                  "tensor_TFLOPs_algorithmic": tflops,
                                  "tensor_frac_of_measured_bf16": (tflops / BF16_PEAK[0]) if BF16_PEAK[0] else None,
                                  "D_mse": d_mse, "D_prod": d_prod}
        res[f"{bits - 1}+1bit"]["GB_s_frac_of_measured_hbm"] = res[f"{bits - 1}+1bit"]["GB_s"] / peaks()[0]
        del out
    return {"workload": "32 layers x 8 KV heads x 16384 tokens x d=128 bf16", **res}


def _decode_split(ctx, codes, Pi, cent_lo, cent_hi):
    """x_hat of split codes (flat rows of ctx.row_words words), in torch (measurement only)."""
    words = codes.planes.view(torch.int32).long() & 0xFFFFFFFF
    n = words.shape[0]
    W, P = ctx.W, ctx.P
    j = torch.arange(ctx.d, device=words.device)
    idx = torch.zeros(n, ctx.d, dtype=torch.long, device=words.device)
    for p in range(P):
        idx |= ((words[:, p * W + j // 32] >> (j % 32)) & 1) << p
    hi = j < ctx.d_hi
    jt = torch.clamp(j, max=max(ctx.d_hi - 1, 0))
    top = ((words[:, P * W + jt // 32] >> (jt % 32)) & 1) * hi
    idx |= top << P
    c = torch.where(hi[None, :], cent_hi[idx.clamp(max=len(cent_hi) - 1)], cent_lo[idx.clamp(max=len(cent_lo) - 1)])
    nrm = codes.norm.view(torch.float16).float()
    return nrm[:, None] * (c @ Pi)


def measure_fractional(dev):
    """Fractional bit widths (split contexts): 3.5 and 2.5 bits per channel = 2 / 1 MSE bits with
    the first half of the rotated coordinates one bit higher, plus 1 QJL bit.  Keys of the
    decode-layer shape at batch 8 (8 x 8 KV heads x 32768 tokens, d=128, bf16 anisotropic)
    quantized on the GPU, then one logits pass of 32 query heads; D_mse and D_prod as in the
    prefill workload."""
    from compressed_kv_cache_02_b300 import inputs, tq
    Bf, Hf, Nf, Gf = 8, 8, 32768, 4
    n = Bf * Hf * Nf
    fac = inputs.anisotropic_factors(Hf, D, seed=2, device=dev)
    X = inputs.anisotropic(Bf, Hf, Nf, D, fac, seed=2, device=dev)
    q = inputs.anisotropic(Bf, Hf, Gf, D, fac, seed=2002, device=dev, dtype=torch.float32).reshape(Bf, Hf * Gf, D)
    Qs = q.reshape(-1, D)
    g = torch.Generator(device=dev)
    g.manual_seed(8)
    sample = torch.randperm(n, generator=g, device=dev)[: 1 << 16]
    length = torch.full((Bf,), Nf, dtype=torch.int32, device=dev)
    res = {}
    for label, bits in (("3.5bit", 3), ("2.5bit", 2)):
        ctx = tq.Context(D, bits, seed=0, d_hi=D // 2)
        keys = ctx.alloc_codes(Bf, Hf, Nf, device=dev)
        flat = tq.Codes(keys.planes.view(n, -1), keys.norm.view(n), keys.signs.view(n, -1), keys.rnorm.view(n))
        ctx.quantize(X.reshape(n, D), out=flat)
        tq_q, _ = _event_time(lambda: ctx.quantize(X.reshape(n, D), out=flat))
        ws = ctx.attn_workspace(Bf, Hf * Gf, Hf, Nf, device=dev)
        logits = torch.empty(Bf, Hf * Gf, Nf, device=dev)
        scale = 1.0 / D ** 0.5
        ctx.attn_logits(q, keys, Nf, length, scale, out=logits, workspace=ws)
        t_l, _ = _event_time(lambda: ctx.attn_logits(q, keys, Nf, length, scale, out=logits, workspace=ws), reps=5)
        if ctx.sync_status():
            raise RuntimeError("device error flags in the fractional workload")
        Pi, _, cent_lo, _ = ctx.export()
        cent_hi, _ = tq.host_codebook(D, ctx.P + 1)
        Pi_t = torch.from_numpy(Pi).to(dev)
        xs = X.reshape(n, D)[sample].float()
        sub = tq.Codes(flat.planes[sample], flat.norm[sample], flat.signs[sample], flat.rnorm[sample])
        xh = _decode_split(ctx, sub, Pi_t, torch.from_numpy(cent_lo).float().to(dev),
                           torch.from_numpy(cent_hi).float().to(dev))
        d_mse = float(((xs - xh) ** 2).sum(1).div(xs.pow(2).sum(1)).mean())
        ks = 1 << 14
        sk = tq.Codes(sub.planes[:ks].reshape(1, 1, ks, -1), sub.norm[:ks].reshape(1, 1, ks),
                      sub.signs[:ks].reshape(1, 1, ks, -1), sub.rnorm[:ks].reshape(1, 1, ks))
        Q1 = Qs[:256]
        est = ctx.attn_logits(Q1.reshape(1, 256, D), sk, ks, torch.tensor([ks], dtype=torch.int32, device=dev), 1.0)[0]
        exact = Q1 @ xs[:ks].T
        den = Q1.pow(2).sum(1)[:, None] * xs[:ks].pow(2).sum(1)[None, :]
        d_prod = float(((est - exact) ** 2 / den).mean())
        key_bytes = (ctx.row_words + ctx.Ws) * 4 + 4
        logit_bytes = n * (key_bytes + Gf * 4)
        hbm, _ = peaks()
        # values at the same fractional width (MSE: bits + 0.5 per channel), softmax + value sum
        vbits = bits   # the same width as the keys: 3.5 (2.5) bits per value channel
        vctx = tq.Context(D, vbits, seed=1, mode=tq.TQ_MODE_MSE, d_hi=D // 2)
        vals = vctx.alloc_codes(Bf, Hf, Nf, device=dev)
        Vx = inputs.anisotropic(Bf, Hf, Nf, D, inputs.anisotropic_factors(Hf, D, seed=1002, device=dev), seed=1002,
                                device=dev)
        vctx.quantize(Vx.reshape(n, D), out=tq.Codes(vals.planes.view(n, -1), vals.norm.view(n)))
        del Vx
        vws = tq.values_workspace(D, Bf, Hf * Gf, Hf, Nf, device=dev)
        vout = torch.empty(Bf, Hf * Gf, D, device=dev)
        tq.attn_values(logits, length, vals, vctx=vctx, out=vout, workspace=vws)
        t_v, _ = _event_time(lambda: tq.attn_values(logits, length, vals, vctx=vctx, out=vout, workspace=vws), reps=5)
        if vctx.sync_status():
            raise RuntimeError("device error flags in the fractional values")
        res[label] = {"mse_bits": ctx.P + 0.5, "code_bytes_per_key": key_bytes, "quantize_ms": tq_q * 1e3,
                      "vectors_per_s": n / tq_q, "logits_ms": t_l * 1e3, "logit_scores_per_s": n * Gf / t_l,
                      "logits_GB_s": logit_bytes / t_l / 1e9, "logits_frac_of_measured_hbm": logit_bytes / t_l / 1e9 / hbm,
                      "D_mse": d_mse, "D_prod": d_prod,
                      "values_mse_bits": vbits + 0.5, "values_ms": t_v * 1e3,
                      "attention_ms": (t_l + t_v) * 1e3}
        del keys, flat, logits, ws, vals, vws, vout
    return {"workload": "8 x 8 KV heads x 32768 keys d=128 bf16, 32 query heads; first 64 rotated coordinates +1 bit",
            **res}


def measure_decode1(dev):
    """One decode layer of an 8B-class GQA model at batch 1: 8 KV heads x 32768 tokens, d=128,
    32 query heads; keys bf16 anisotropic coded at 4 bits (3 MSE + 1 QJL), values bf16.  All keys
    are quantized, then the step (rotated queries, logits, softmax and the bf16 value sum:
    tq_attn_output) runs 1000 times eagerly and 1000 times as one captured CUDA graph; the step
    moves ~85 MB, so launch latency matters and the graph removes it."""
    from compressed_kv_cache_02_b300 import inputs, tq
    hkv, n, g, seed = 8, 32768, 4, 2
    ctx = tq.Context(D, 4, seed=0)
    kfac = inputs.anisotropic_factors(hkv, D, seed=seed, device=dev)
    vfac = inputs.anisotropic_factors(hkv, D, seed=seed + 1000, device=dev)
    K = inputs.anisotropic(1, hkv, n, D, kfac, seed=seed, device=dev)
    V = inputs.anisotropic(1, hkv, n, D, vfac, seed=seed + 1000, device=dev)
    q = inputs.anisotropic(1, hkv, g, D, kfac, seed=seed + 2000, device=dev, dtype=torch.float32).reshape(1, hkv * g, D)
    kc = ctx.alloc_codes(1, hkv, n, device=dev)
    flat = tq.Codes(kc.planes.view(hkv * n, ctx.P, -1), kc.norm.view(-1), kc.signs.view(hkv * n, -1), kc.rnorm.view(-1))
    ctx.quantize(K.reshape(hkv * n, D), out=flat)
    t_q, _ = _event_time(lambda: ctx.quantize(K.reshape(hkv * n, D), out=flat), reps=10)
    length = torch.tensor([n], dtype=torch.int32, device=dev)
    scale = 1.0 / D ** 0.5
    ws = ctx.attn_workspace(1, hkv * g, hkv, n, device=dev)
    out = torch.empty(1, hkv * g, D, device=dev)
    logits = torch.empty(1, hkv * g, n, device=dev)

    def step():
        ctx.attn_output(q, kc, n, length, scale, V, out=out, workspace=ws)

    for _ in range(20):
        step()
    reps = 1000
    t_eager, _ = _event_time(step, reps=reps)
    t_logits, _ = _event_time(lambda: ctx.attn_logits(q, kc, n, length, scale, out=logits, workspace=ws), reps=reps)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    t_graph, _ = _event_time(graph.replay, reps=reps)
    # the step's 85 MB fit in L2: also time it cold, after writing a 256 MB buffer each time
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    for e0, e1 in evs:
        flush.fill_(1)
        e0.record()
        graph.replay()
        e1.record()
    torch.cuda.synchronize()
    t_cold = sum(e0.elapsed_time(e1) for e0, e1 in evs) / len(evs) / 1e3
    del flush
    if ctx.sync_status():
        raise RuntimeError("device error flags in the batch-1 decode workload")
    keys = hkv * n
    key_bytes = (ctx.P * ctx.W + ctx.Ws) * 4 + 4
    step_bytes = keys * (key_bytes + 2 * D)   # codes + bf16 values read once
    logit_bytes = keys * (key_bytes + g * 4)
    hbm, _ = peaks()
    return {"workload": "batch 1, 8 KV heads x 32768 tokens, d=128, 32 query heads; keys 4-bit (3+1), values bf16",
            "quantize_keys_ms": t_q * 1e3, "quantize_vectors_per_s": keys / t_q,
            "l2": "step inputs (85 MB) fit in L2: step_ms_graph repeats L2-warm; step_ms_graph_cold after a 256 MB write",
            "step_ms_eager": t_eager * 1e3, "step_ms_graph": t_graph * 1e3, "step_ms_graph_cold": t_cold * 1e3,
            "step_GB_s_graph_cold": step_bytes / t_cold / 1e9,
            "step_frac_of_measured_hbm_graph_cold": step_bytes / t_cold / 1e9 / hbm,
            "logit_scores_per_s_graph": keys * g / t_graph, "step_GB_s_graph": step_bytes / t_graph / 1e9,
            "step_frac_of_measured_hbm_graph": step_bytes / t_graph / 1e9 / hbm,
            "logits_ms": t_logits * 1e3, "logits_GB_s": logit_bytes / t_logits / 1e9,
            "bytes_per_step": step_bytes, "repeats": reps}


def measure_paged(dev, steps=16, warmup=3, state=None):
    """The headline decode workload (batch 8, 8 KV heads x 131072 cached tokens, keys 2+1 bits,
    values 3-bit MSE) over a paged cache: pages of 256 tokens placed at random in the pools
    through the block table, each step one fused persistent launch (append + logits + softmax +
    values + merge + advance: tq_paged_decode_step).  Inputs (~0.9 GB of pools) exceed L2."""
    from compressed_kv_cache_02_b300 import tq
    st = build_state(dev) if state is None else state
    kctx, vctx, kc, vc, cap = st["kctx"], st["vctx"], st["kc"], st["vc"], st["cap"]
    ps = 256
    npp = cap // ps
    num_pages = B * npp
    g = torch.Generator(device="cpu")
    g.manual_seed(11)
    perm = torch.randperm(num_pages, generator=g).to(dev)

    def pool(x):   # [B, Hkv, cap, ...] -> [num_pages, Hkv, ps, ...], page (b, i) at perm[b * npp + i]
        rest = x.shape[3:]
        ordered = x.reshape(B, HKV, npp, ps, *rest).transpose(1, 2).reshape(num_pages, HKV, ps, *rest)
        out = torch.empty_like(ordered)
        out[perm] = ordered
        return out

    cache = tq.PagedCache(kplanes=pool(kc.planes), ksigns=pool(kc.signs), knorm=pool(kc.norm),
                          krnorm=pool(kc.rnorm), vplanes=pool(vc.planes), vnorm=pool(vc.norm))
    del kc, vc, st["kc"], st["vc"]
    table = perm.reshape(B, npp).to(torch.int32).contiguous()
    length = torch.full((B,), N0, dtype=torch.int32, device=dev)
    ks, vs, qs = step_inputs(st, warmup + steps, dev)
    scale = 1.0 / D ** 0.5
    ws = tq.paged_workspace(B, HQ, HKV, npp, ps, device=dev)
    out = torch.empty(B, HQ, D, device=dev)
    for s_ in range(warmup):
        tq.paged_decode_step(kctx, vctx, qs[s_], ks[s_], vs[s_], cache, table, length, scale, out=out, workspace=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s_ in range(warmup, warmup + steps):
        tq.paged_decode_step(kctx, vctx, qs[s_], ks[s_], vs[s_], cache, table, length, scale, out=out, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / steps
    flags = kctx.sync_status()
    if flags:
        raise RuntimeError(f"device error flags {flags} in the paged workload")
    keys = B * HKV * (N0 + warmup + steps / 2)
    step_bytes = keys * (K_BYTES + V_BYTES)
    hbm, _ = peaks()
    del cache, ks, vs, qs, st
    torch.cuda.empty_cache()
    return {"workload": WORKLOAD + "; paged cache (256-token pages, random placement), one fused launch per step",
            "steps": steps, "ms_per_step": t * 1e3, "logit_scores_per_s": keys * G / t,
            "step_GB_s": step_bytes / t / 1e9, "step_frac_of_measured_hbm": step_bytes / t / 1e9 / hbm,
            "bytes_per_key": K_BYTES + V_BYTES, "launches_per_step": 1,
            "batch1": measure_paged_small(dev)}


def measure_paged_small(dev, reps=200):
    """Latency-bound size for the fused step: batch 1, 8 KV heads x 32768 cached tokens, keys 2+1
    bits, values 3-bit MSE.  The fused paged step (one launch) against the unfused step on the
    same codes (key and value appends, advance, logits, values + combine: 8 launches), each
    repeated `reps` times back to back (the cache, ~27 MB, stays in L2 in both)."""
    from compressed_kv_cache_02_b300 import inputs, tq
    b1, n0, ps = 1, 32768, 256
    kctx = tq.Context(D, KBITS, seed=SEED_ROT)
    vctx = tq.Context(D, VBITS, seed=SEED_ROT + 1, mode=tq.TQ_MODE_MSE)
    cap = n0 + 2 * reps + 1024
    cap = ((cap + ps - 1) // ps) * ps
    kfac = inputs.anisotropic_factors(HKV, D, seed=SEED_DATA, device=dev)
    vfac = inputs.anisotropic_factors(HKV, D, seed=SEED_DATA + 1000, device=dev)
    K = inputs.anisotropic(b1, HKV, n0, D, kfac, seed=SEED_DATA * 100, device=dev)
    V = inputs.anisotropic(b1, HKV, n0, D, vfac, seed=SEED_DATA * 100 + 1000, device=dev)
    kc = kctx.alloc_codes(b1, HKV, cap, device=dev)
    vc = vctx.alloc_codes(b1, HKV, cap, device=dev)
    for h in range(HKV):
        kctx.quantize(K[0, h], out=tq.Codes(kc.planes[0, h, :n0], kc.norm[0, h, :n0], kc.signs[0, h, :n0],
                                            kc.rnorm[0, h, :n0]))
        vctx.quantize(V[0, h], out=tq.Codes(vc.planes[0, h, :n0], vc.norm[0, h, :n0]))
    kn = inputs.anisotropic(b1, HKV, 1, D, kfac, seed=10_001, device=dev)[:, :, 0].contiguous()
    vn = inputs.anisotropic(b1, HKV, 1, D, vfac, seed=20_001, device=dev)[:, :, 0].contiguous()
    q = inputs.anisotropic(b1, HKV, G, D, kfac, seed=30_001, device=dev, dtype=torch.float32).reshape(b1, HQ, D)
    scale = 1.0 / D ** 0.5
    # unfused: the headline step's calls on this cache
    length = torch.full((b1,), n0, dtype=torch.int32, device=dev)
    logits = torch.empty(b1, HQ, cap, device=dev)
    out = torch.empty(b1, HQ, D, device=dev)
    ws = kctx.attn_workspace(b1, HQ, HKV, cap, device=dev)
    vws = tq.values_workspace(D, b1, HQ, HKV, cap, device=dev)

    def unfused():
        kctx.append(kn, kc, cap, length)
        vctx.append(vn, vc, cap, length)
        kctx.advance_len(length, cap)
        kctx.attn_logits(q, kc, cap, length, scale, out=logits, workspace=ws)
        tq.attn_values(logits, length, vc, vctx=vctx, out=out, workspace=vws)

    for _ in range(5):
        unfused()
    t_unf, _ = _event_time(unfused, reps=reps)
    # fused: the same codes in pages (identity placement)
    npp = cap // ps

    def pool(x):
        rest = x.shape[3:]
        return x.reshape(b1, HKV, npp, ps, *rest).transpose(1, 2).reshape(b1 * npp, HKV, ps, *rest).contiguous()

    cache = tq.PagedCache(kplanes=pool(kc.planes), ksigns=pool(kc.signs), knorm=pool(kc.norm), krnorm=pool(kc.rnorm),
                          vplanes=pool(vc.planes), vnorm=pool(vc.norm))
    table = torch.arange(npp, dtype=torch.int32, device=dev).reshape(b1, npp)
    plen = torch.full((b1,), n0, dtype=torch.int32, device=dev)
    pws = tq.paged_workspace(b1, HQ, HKV, npp, ps, device=dev)

    def fused():
        tq.paged_decode_step(kctx, vctx, q, kn, vn, cache, table, plen, scale, out=out, workspace=pws)

    for _ in range(5):
        fused()
    t_fus, _ = _event_time(fused, reps=reps)
    if kctx.sync_status() or vctx.sync_status():
        raise RuntimeError("device error flags in the small paged workload")
    return {"workload": "batch 1, 8 KV heads x 32768 tokens, d=128, 32 query heads; keys 2+1 bits, values 3-bit MSE",
            "step_ms_unfused": t_unf * 1e3, "launches_unfused": 8, "step_ms_fused_paged": t_fus * 1e3,
            "launches_fused": 1, "repeats": reps, "l2": "cache ~27 MB, L2-resident in both arms"}


def _decode_polar(pc, d, bits, Pi_t, tables):
    """x_hat of polar codes on the device (measurement only): unpack the b-bit fields, rebuild
    y_hat top-down from r16 and the per-level angle centroids, rotate back."""
    n = pc.codes.shape[0]
    w = pc.codes.view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    bitsm = (w.unsqueeze(-1) >> torch.arange(32, device=w.device)) & 1
    stream = bitsm.reshape(n, -1)[:, :(d - 1) * bits].reshape(n, d - 1, bits)
    codes = (stream << torch.arange(bits, device=w.device)).sum(-1)
    r = pc.r16.view(torch.float16).float()
    levels, a, width = [], 0, d // 2
    while width >= 1:
        levels.append(codes[:, a:a + width])
        a += width
        width //= 2
    cur = r[:, None]
    for lev in range(len(levels), 0, -1):
        ang = tables[lev - 1][levels[lev - 1]]
        out = torch.empty(n, 2 * cur.shape[1], device=cur.device)
        out[:, 0::2] = cur * torch.cos(ang)
        out[:, 1::2] = cur * torch.sin(ang)
        cur = out
    return cur @ Pi_t


def measure_polar(dev):
    """Polar-angle encoder (r16 + d - 1 angles of b bits + 1 QJL bit): keys of the decode-layer
    shape at batch 8 (8 x 8 KV heads x 32768 tokens, d=128, bf16 anisotropic) quantized on the
    GPU; scores of one 4-query group against every key; D_mse on a 65536-key sample and D_prod
    of 256 queries x 16384 keys, as in the prefill workload."""
    from compressed_kv_cache_02_b300 import inputs, tq
    Bf, Hf, Nf, Gf = 8, 8, 32768, 4
    n = Bf * Hf * Nf
    fac = inputs.anisotropic_factors(Hf, D, seed=2, device=dev)
    X = inputs.anisotropic(Bf, Hf, Nf, D, fac, seed=2, device=dev).reshape(n, D)
    q = inputs.anisotropic(Bf, Hf, Gf, D, fac, seed=2002, device=dev, dtype=torch.float32).reshape(-1, D)
    g = torch.Generator(device=dev)
    g.manual_seed(8)
    sample = torch.randperm(n, generator=g, device=dev)[: 1 << 16]
    Pi, _ = tq.host_matrices(0, D, D)
    Pi_t = torch.from_numpy(Pi).to(dev)
    hbm, _ = peaks()
    res = {}
    for label, bits in (("4bit_standard", 3), ("3bit_extreme", 2)):
        ctx = tq.PolarContext(D, bits, qjl=True, seed=0)
        pc = ctx.alloc_codes(n, device=dev)
        ctx.quantize(X, out=pc)
        ctx.set_kernel_path(tq.TQ_PATH_CUDA_CORE)   # the CUDA-core encoder, for comparison
        ctx.quantize(X, out=pc)
        t_qc, _ = _event_time(lambda: ctx.quantize(X, out=pc))
        ctx.set_kernel_path(tq.TQ_PATH_AUTO)        # tcgen05 for these bf16 rows at d = 128
        ctx.quantize(X, out=pc)
        t_q, _ = _event_time(lambda: ctx.quantize(X, out=pc))
        out = torch.empty(Gf, n, device=dev)
        ctx.scores(q[:Gf], pc, 1.0, out=out)
        t_s, _ = _event_time(lambda: ctx.scores(q[:Gf], pc, 1.0, out=out), reps=5)
        if ctx.sync_status():
            raise RuntimeError("device error flags in the polar workload")
        tables = [torch.from_numpy(tq.host_polar_codebook(lev, bits)[0]).float().to(dev) for lev in range(1, 8)]
        xs = X[sample].float()
        sub = tq.PolarCodes(pc.codes[sample], pc.r16[sample], pc.signs[sample], pc.rnorm[sample])
        xh = _decode_polar(sub, D, bits, Pi_t, tables)
        d_mse = float(((xs - xh) ** 2).sum(1).div(xs.pow(2).sum(1)).mean())
        ks = 1 << 14
        sk = tq.PolarCodes(sub.codes[:ks].contiguous(), sub.r16[:ks].contiguous(), sub.signs[:ks].contiguous(),
                           sub.rnorm[:ks].contiguous())
        Q1 = q[:256]
        est = ctx.scores(Q1, sk, 1.0)
        exact = Q1 @ xs[:ks].T
        den = Q1.pow(2).sum(1)[:, None] * xs[:ks].pow(2).sum(1)[None, :]
        d_prod = float(((est - exact) ** 2 / den).mean())
        key_bytes = (ctx.code_words + ctx.sign_words) * 4 + 4
        score_bytes = n * (key_bytes + Gf * 4)
        res[label] = {"angle_bits": bits, "code_bytes_per_key": key_bytes, "quantize_ms": t_q * 1e3,
                      "quantize_ms_cuda_core": t_qc * 1e3, "vectors_per_s": n / t_q,
                      "quantize_GB_s": n * (D * 2 + key_bytes) / t_q / 1e9, "scores_ms": t_s * 1e3, "scores_per_s": n * Gf / t_s,
                      "scores_GB_s": score_bytes / t_s / 1e9, "scores_frac_of_measured_hbm": score_bytes / t_s / 1e9 / hbm,
                      "D_mse": d_mse, "D_prod": d_prod}
        del pc, out, ctx
    return {"workload": "8 x 8 KV heads x 32768 keys d=128 bf16 (2.1M vectors); polar r16 + 127 angles + 128 QJL bits",
            **res}


# ----------------------------------------------------------------------------- the oracle arm

_PREFILL = {}


def _oracle_group(n_keys: int, seed: int):
    """The oracle's tables, one (batch, KV head) group's coded cache of n_keys keys and values, the
    step's new key and value and its 4 query heads (prepared once per process, not timed)."""
    import oracle
    from compressed_kv_cache_02_b300 import inputs
    key = (n_keys, seed)
    if key not in _PREFILL:
        Pi, S = oracle.method_matrices(SEED_ROT, D, D)
        Piv, _ = oracle.method_matrices(SEED_ROT + 1, D, 1)
        cbk = oracle.sphere_codebook(D, KBITS - 1)
        cbv = oracle.sphere_codebook(D, VBITS)
        fk = inputs.anisotropic_factors(1, D, seed=seed)
        fv = inputs.anisotropic_factors(1, D, seed=seed + 1000)
        K = inputs.anisotropic(1, 1, n_keys + 1, D, fk, seed=seed).float().numpy()
        V = inputs.anisotropic(1, 1, n_keys + 1, D, fv, seed=seed + 1000).float().numpy()
        q = inputs.anisotropic(1, 1, G, D, fk, seed=seed + 2000, dtype=torch.float32).numpy().reshape(1, G, D)
        kz = oracle.quantize(K[0, 0, :n_keys], Pi, cbk, S)
        vz = oracle.quantize(V[0, 0, :n_keys], Piv, cbv)
        _PREFILL[key] = (Pi, S, Piv, cbk, cbv, K, V, q, kz, vz)
    return _PREFILL[key]


def oracle_step_sample(n_keys: int, seed: int = SEED_DATA):
    """Bounded oracle sample of one decode step: one (batch, KV head) group with n_keys cached
    keys and values, its 4 query heads: quantize the new key and value, score every key (the
    logits, once) and form the softmax-weighted sum of the values.  Returns (logit scores
    computed, seconds)."""
    import oracle
    Pi, S, Piv, cbk, cbv, K, V, q, kz, vz = _oracle_group(n_keys, seed)
    t = time.perf_counter()
    kn = oracle.quantize(K[0, 0, n_keys:], Pi, cbk, S)          # the step's append
    vn = oracle.quantize(V[0, 0, n_keys:], Piv, cbv)
    keys = oracle.Quantized(idx=np.concatenate([kz.idx, kn.idx])[None, None],
                            norm16=np.concatenate([kz.norm16, kn.norm16])[None, None],
                            signs=np.concatenate([kz.signs, kn.signs])[None, None],
                            rnorm16=np.concatenate([kz.rnorm16, kn.rnorm16])[None, None])
    vals = oracle.Quantized(idx=np.concatenate([vz.idx, vn.idx])[None, None],
                            norm16=np.concatenate([vz.norm16, vn.norm16])[None, None])
    L = np.array([n_keys + 1])
    logits = oracle.attention_logits(q, keys, L, Pi, S, cbk, 1.0 / D ** 0.5)
    oracle.attention_values(logits, L, 1, values=vals, Pi_v=Piv, cb_v=cbv)
    return G * (n_keys + 1), time.perf_counter() - t


def _oracle_worker_init():
    torch.set_num_threads(1)


def _oracle_job(job):
    """One worker's share: prepare its group (untimed), then samples for about budget_s seconds
    (at least one, at most max_reps).  Returns (scores, wall start, wall end, samples, pid)."""
    n_keys, seed, budget_s, max_reps = job
    _oracle_group(n_keys, seed)
    done, reps = 0, 0
    t0 = time.time()
    while (reps == 0 or time.time() - t0 < budget_s) and reps < max_reps:
        s, _ = oracle_step_sample(n_keys, seed)
        done += s
        reps += 1
    return done, t0, time.time(), reps, os.getpid()


class OraclePool:
    """The oracle on every host core this process may use: one spawned worker per core (spawned,
    since the parent has already used the GPU), each single-threaded (BLAS and torch), each
    decoding its own (batch, KV head) group.  Throughput = all workers' logit scores / the wall
    span from the first worker's start to the last one's end."""

    MAX_WORKERS = 128

    def __init__(self, n_keys: int = 32768):
        import concurrent.futures as cf
        import multiprocessing as mp
        self.n_keys = n_keys
        self.host_cores = len(os.sched_getaffinity(0))
        self.workers = min(self.host_cores, self.MAX_WORKERS)
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.ex = cf.ProcessPoolExecutor(self.workers, mp_context=mp.get_context("spawn"),
                                             initializer=_oracle_worker_init)
            self.run(0.0, 1)   # start the workers and prepare their groups
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def run(self, budget_s: float, max_reps: int):
        jobs = [(self.n_keys, SEED_DATA + w, budget_s, max_reps) for w in range(self.workers)]
        res = list(self.ex.map(_oracle_job, jobs))
        scores = sum(r[0] for r in res)
        span = max(r[2] for r in res) - min(r[1] for r in res)
        return scores, span, sum(r[3] for r in res), len({r[4] for r in res})

    def close(self):
        self.ex.shutdown()


def cpu_baseline(args, budget_s: float = 15.0):
    pool = OraclePool()
    try:
        scores, span, reps, used = pool.run(budget_s, 10_000)
    finally:
        pool.close()
    return {"value": scores / span, "unit": UNIT, "cores": used, "host_cores": pool.host_cores, "kind": "oracle",
            "sample": f"{reps} one-group decode steps over {used} single-threaded worker processes (one per core, "
                      f"~{budget_s:.0f} s each): append + logits + softmax-weighted values of 4 query heads x "
                      f"{pool.n_keys + 1} cached keys, numpy float64; scores / wall span of all workers"}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    pool = OraclePool()
    try:
        for _ in range(args.warmup):
            pool.run(0.0, 1)
        done, spent, reps, used = 0, 0.0, 0, 0
        for _ in range(args.steps):
            s, t, r, u = pool.run(0.0, 1)
            done += s
            spent += t
            reps += r
            used = max(used, u)
    finally:
        pool.close()
    v = done / spent
    sample = (f"each step: every worker process ({used}, one per host core) decodes one (batch, KV head) group of "
              f"the decode workload, 4 query heads x {pool.n_keys + 1} cached keys (append + logits + values), "
              f"numpy float64 oracle; step time = wall span of the workers")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": spent / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": used, "host_cores": pool.host_cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["tq", "reference"], default="tq")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-extra", action="store_true", help="skip the search and prefill workloads")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--batch", type=int, default=B, help="smaller batch for profiling captures (default 8)")
    ap.add_argument("--kernel-path", choices=["auto", "cuda_core", "tensor"], default="auto",
                    help="kernel family of the decode step (tq_set_kernel_path)")
    ap.add_argument("--values-path", choices=["auto", "cuda_core", "tensor"], default=None,
                    help="kernel family of the value sum (default: --kernel-path)")
    ap.add_argument("--only", choices=["search", "prefill", "fractional", "polar", "decode1", "paged"], default=None,
                    help="run only one secondary workload and print its measurements (profiling captures)")
    args = ap.parse_args()
    set_batch(args.batch)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.only:
        torch.cuda.set_device(local)
        fn = {"search": measure_search, "prefill": measure_prefill, "fractional": measure_fractional,
              "polar": measure_polar, "decode1": measure_decode1, "paged": measure_paged}[args.only]
        print(json.dumps({"only": args.only, **fn(torch.device("cuda", local))}), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_tq(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
