"""Benchmark of the exact-attention hot path (forward + backward) on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = fa_fwd then fa_bwd (its three stages) over one batch of the
workload, inputs resident in HBM, captured once into a CUDA graph and timed
as one replay per step (`--eager`: as eager calls); per-kernel times and the
roofline come from eager calls with CUDA events between the kernels.
`value` is algorithmic TFLOPS (forward
4 B H N^2 d, backward 2.5x that, halved for causal; block-sparse counts the
kept blocks), summed over ranks under torchrun (each rank runs the whole
workload on its own GPU: weak scaling, no collective on the data path).
L2 is flushed (a 256 MiB write) between timed steps, outside the timed events.
`e2e` is the same metric through the public binding with pinned host inputs
copied in and every output copied back inside the timed region.
`--impl reference` times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

# BLAS threads for the CPU oracle: every core this process may run on.
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPS (bf16, 1×GB300) and % of dense tensor-core peak"
UNIT = "TFLOPS"
DEFAULT_WORKLOAD = "fwdbwd_b2h16n4096d128_causal"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return PEAKS_FALLBACK, "fallback"


# tcgen05 bf16 rate of one SM, measured on this GPU with a microbenchmark of
# back-to-back 128 x 128 x 16 MMAs: 64 cycles each, i.e. 8192 FLOP per clock.
BF16_FLOP_PER_CLK_PER_SM = 8192


def _other_peaks(achieved, peaks, clocks, dev):
    """The achieved rate against the measured sustained peak and against the
    theoretical peak at the median SM clock of the timed region."""
    import torch
    out = {}
    if "bf16_tflops_sustained" in peaks:
        ps = float(peaks["bf16_tflops_sustained"])
        out["sustained"] = {"peak": ps, "frac": achieved / ps, "source": "measured bf16 dense (sustained)"}
    try:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = float(clocks["sm_mhz"]) if clocks and clocks.get("sm_mhz") else None
        if mhz:
            pt = BF16_FLOP_PER_CLK_PER_SM * sms * mhz * 1e6 / 1e12
            out["theoretical_at_clock"] = {"peak": pt, "frac": achieved / pt, "sms": sms, "sm_mhz": mhz,
                                           "source": "8192 FLOP/clk/SM (measured MMA rate) x SMs x median clock"}
    except Exception:
        pass
    return out


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world_size: int, flops_per_rank_step: float, ms_per_step: float) -> float:
    """Weak scaling: every rank runs the whole workload, so the job does
    world_size times the work of one rank in the slowest rank's time."""
    return world_size * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def _count_flops(B, H, N, d, causal=False, backward=False, density=None) -> float:
    """The FLOP convention of the measurements: 4 B H N^2 d forward (two N x N
    x d products), 2.5x that backward (five products), halved when causal,
    scaled by the kept fraction of a block mask."""
    f = 4.0 * B * H * N * N * d
    if backward:
        f *= 2.5
    if causal:
        f *= 0.5
    if density is not None:
        f *= density
    return f


def _flops(w, density):
    """With a block mask, `density` already carries the causal halving (see
    _density), so the causal factor is applied only without one."""
    causal = w.causal and density is None
    f_fwd = _count_flops(w.B, w.H, w.N, w.d, causal=causal, density=density)
    f_bwd = _count_flops(w.B, w.H, w.N, w.d, causal=causal, backward=True, density=density) if w.backward else 0.0
    return f_fwd, f_bwd


def _decode_pairs(nq, L, causal):
    """(query, key) pairs a decode step scores: query i of nq sits at position
    L - nq + i of a cache of L rows; causal keeps keys up to that position."""
    if not causal:
        return nq * L
    return sum(min(max(L - nq + i + 1, 0), L) for i in range(nq))


def _decode_work(w, seqlens):
    """(FLOPs, cache bytes read) of one decode step: 4 d FLOPs per pair, and K
    and V rows of every valid cache position read once per (batch, head)."""
    pairs = sum(_decode_pairs(w.nq, int(L), w.causal) for L in seqlens) * w.H
    cache_bytes = sum(int(L) for L in seqlens) * w.H * w.d * 2 * 2
    io_bytes = w.B * w.H * w.nq * (w.d * 2 * 2 + 4)       # q in, o and lse out
    return 4.0 * w.d * pairs, cache_bytes + io_bytes


def _density(t, causal=False):
    """Fraction of the N x N scores a block mask keeps.  With the causal flag,
    blocks above the diagonal count 0 and diagonal blocks 1/2, the same
    halving as the causal FLOP convention (all blocks kept -> exactly 1/2)."""
    import torch
    bm = t.get("block_mask")
    if bm is None:
        return None
    m = bm.float()
    if not causal:
        return float(m.mean())
    return float((torch.tril(m, -1).sum() + 0.5 * torch.diagonal(m).sum()) / m.numel())


def _config(w, density, extra=None):
    c = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
         "mask": w.mask_kind, "backward": w.backward, "inputs": f"N(0,1)x{w.amplitude:g} seed {w.seed}",
         "l2": "flushed (256 MiB write) between timed steps", "parallelism": "replica per GPU"}
    if density is not None:
        c["block_density"] = round(density, 4)
    if getattr(w, "dropout_p", 0.0):
        c["dropout_p"] = w.dropout_p
    if extra:
        c.update(extra)
    return c


# --------------------------------------------------------------------------- #
# clocks during the timed region
# --------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and self.uuid not in parts[1]:
                    continue
                try:
                    rows.append({"sm": float(parts[2]), "max": float(parts[3]), "power": float(parts[4]),
                                 "hw": parts[6], "hw_thermal": parts[7], "sw_thermal": parts[8], "power_cap": parts[9]})
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("power_cap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r["power"] for r in rows)}


# --------------------------------------------------------------------------- #
# the CPU oracle on a bounded sample
# --------------------------------------------------------------------------- #
class Parity:
    """Comparison of the timed step's outputs with the oracle's, on the whole
    heads that the CPU-baseline leg runs anyway.  Bounds as in the parity
    tests: O within 1e-2 + 2^-8 |O_ref| element-wise (plus the oracle's bound
    on bf16 probabilities in P V for inputs of amplitude > 1), LSE relative 1e-3
    (against max(|LSE|, 1)), dQ, dK, dV relative L2 2e-2 per head and per
    128-row tile, and (first two heads, no dropout) every gradient element
    inside the oracle's error model, u |r| + (1 + u)(6 sigma + acc); the 8-bit
    forward within the oracle's e4m3 error model plus O's bf16 rounding."""

    def __init__(self):
        self.o_excess = -float("inf")
        self.o_max_abs = 0.0
        self.lse_rel = 0.0
        self.rel = {"dq": 0.0, "dk": 0.0, "dv": 0.0}
        self.tile_rel = 0.0
        self.grad_excess = None
        self.heads = 0
        self.element_heads = 0

    @staticmethod
    def _np(x):
        return x.float().numpy()

    def forward(self, o, lse, ro, rl, bound=None):
        import numpy as np
        o, lse = self._np(o), self._np(lse)
        lim = (1e-2 + 2.0 ** -8 * np.abs(ro)) if bound is None else bound
        err = np.abs(o - ro)
        self.o_excess = max(self.o_excess, float(np.nanmax(np.where(np.isfinite(o), err - lim, np.inf))))
        self.o_max_abs = max(self.o_max_abs, float(err.max()))
        fin = np.isfinite(rl)
        if not np.array_equal(np.isfinite(lse), fin):
            self.lse_rel = float("inf")
        elif fin.any():
            self.lse_rel = max(self.lse_rel, float((np.abs(lse[fin] - rl[fin]) / np.maximum(np.abs(rl[fin]), 1.0)).max()))

    def backward(self, g, ref, model=None):
        import numpy as np
        for i, (name, a, r) in enumerate(zip(("dq", "dk", "dv"), g, ref)):
            a = self._np(a)
            floor = 1e-3 * np.sqrt(r.size)
            self.rel[name] = max(self.rel[name], float(np.linalg.norm(a - r) / max(np.linalg.norm(r), floor)))
            n = r.shape[-2]
            for t0 in range(0, n, 128):
                x, y = a[..., t0:t0 + 128, :], r[..., t0:t0 + 128, :]
                tr = np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-3 * np.sqrt(y.size))
                self.tile_rel = max(self.tile_rel, float(tr))
            if model is not None:
                u = 2.0 ** -8
                ex = float((np.abs(a - r) - (u * np.abs(r) + (1 + u) * (6 * model[0][i] + model[1][i]))).max())
                self.grad_excess = ex if self.grad_excess is None else max(self.grad_excess, ex)

    def report(self, backward):
        ok = self.heads > 0 and self.o_excess <= 0 and self.lse_rel <= 1e-3
        out = {"heads_checked": self.heads, "o_max_abs": self.o_max_abs, "o_excess": self.o_excess,
               "lse_rel": self.lse_rel}
        if backward:
            out.update({f"{k}_rel_l2": v for k, v in self.rel.items()})
            out["tile_rel_l2"] = self.tile_rel
            ok = ok and max(self.rel.values()) <= 2e-2 and self.tile_rel <= 2e-2
            if self.grad_excess is not None:
                out["grad_element_excess"] = self.grad_excess
                out["grad_element_heads"] = self.element_heads
                ok = ok and self.grad_excess <= 0
        out["ok"] = bool(ok)
        out["source"] = "outputs of the last timed step vs the oracle on the cpu_baseline heads"
        return out


def _oracle_sample(w, t, budget_s=15.0, max_heads=None, gpu=None, parity=None):
    """Time the fp64 oracle (forward + backward) head by head until `budget_s`
    of oracle time has passed.  Returns (TFLOPS, seconds, heads).  With `gpu`
    (the timed step's outputs on the host) and a `parity` accumulator, each
    head's oracle results are also compared with the GPU's, outside the
    timed oracle calls."""
    import oracle
    import torch
    bm = t.get("block_mask")
    bmn = None if bm is None else bm.numpy()
    heads = 0
    flops = 0.0
    el = 0.0
    for hh in range(w.B * w.H):
        b, h = divmod(hh, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        if w.fp8:
            u8 = [t[n][sl].contiguous().view(torch.uint8).numpy() for n in ("q8", "k8", "v8")]
            qd, kd, vd = (t[n][sl].double().numpy() for n in ("qd", "kd", "vd"))
            t0 = time.perf_counter()
            ro, rl, probs, vv = oracle.forward_fp8(*u8, qd, kd, vd, w.scale, causal=w.causal)
            el += time.perf_counter() - t0
            heads += 1
            ff, fb = _flops(type(w)(**{**w.__dict__, "B": 1, "H": 1}), None)
            flops += ff
            if gpu is not None and parity is not None:
                import numpy as np
                bound, _ = oracle.fp8_error_model(ro, probs, vv)
                parity.forward(gpu["o"][sl], gpu["lse"][sl], ro, rl, bound + 2.0 ** -8 * np.abs(ro) + 1e-3)
                parity.heads += 1
            if el >= budget_s or (max_heads and heads >= max_heads):
                break
            continue
        q, k, v = (t[n][sl].double().numpy() for n in ("q", "k", "v"))
        do = t["do"][sl].double().numpy() if w.backward else None
        t0 = time.perf_counter()
        if w.dropout_p:
            ro, rl = oracle.forward_dropout(q, k, v, w.scale, w.dropout_p, w.seed, causal=w.causal, block_mask=bmn,
                                            b0=b, h0=h)
            ref = oracle.backward_dropout(q, k, v, do, w.scale, w.dropout_p, w.seed, causal=w.causal,
                                          block_mask=bmn, b0=b, h0=h)[:3] if w.backward else None
        else:
            ro, rl = oracle.forward(q, k, v, w.scale, causal=w.causal, block_mask=bmn,
                                    row_chunk=2048 if w.N > 8192 else None)
            ref = oracle.backward(q, k, v, do, w.scale, causal=w.causal, block_mask=bmn)[:3] if w.backward else None
        el += time.perf_counter() - t0
        heads += 1
        ff, fb = _flops(type(w)(**{**w.__dict__, "B": 1, "H": 1}), _density(t, w.causal))
        flops += ff + fb
        if gpu is not None and parity is not None:
            limit = None
            if w.amplitude > 1 and not w.dropout_p:
                # inputs of amplitude > 1: add the oracle's bound on the effect of
                # bf16 probabilities in P V, which alone can exceed 1e-2 there
                import numpy as np
                pb = oracle.forward_error_bound(q, k, v, w.scale, causal=w.causal, block_mask=bmn,
                                                row_chunk=2048 if w.N > 8192 else None)
                limit = 1e-2 + 2.0 ** -8 * np.abs(ro) + pb
            parity.forward(gpu["o"][sl], gpu["lse"][sl], ro, rl, limit)
            if w.backward:
                model = None
                if not w.dropout_p and parity.element_heads < 2:
                    model = oracle.grad_error_model(q, k, v, do, w.scale, causal=w.causal, block_mask=bmn)
                    parity.element_heads += 1
                parity.backward([gpu[n][sl] for n in ("dq", "dk", "dv")], ref, model)
            parity.heads += 1
        if el >= budget_s or (max_heads and heads >= max_heads):
            break
    return flops / el / 1e12, el, heads


REF_ROWS = 256   # query rows per reference-arm step


def run_reference(args):
    """The fp64 CPU oracle as the reference arm.  Each step is one block of
    REF_ROWS query rows of head (0, 0): its forward rows (O, LSE) and its part
    of the backward (dQ rows, contributions to dK and dV); successive steps
    walk through the head's row blocks.  Throughput counts the algorithmic
    FLOPs of the visible (query, key) pairs of those rows: 4 d per pair
    forward, 2.5x that backward."""
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import numpy as np
    import torch
    import oracle
    from attn_fwd_gb300.inputs import DECODE_WORKLOADS, WORKLOADS, make_workload_inputs
    if args.workload in DECODE_WORKLOADS:
        return _run_reference_decode(args, DECODE_WORKLOADS[args.workload])
    w = WORKLOADS[args.workload]
    t = make_workload_inputs(w, heads=slice(0, 1))
    if w.fp8:      # the real inputs: e4m3 values times their descales
        q, k, v = (oracle.e4m3_decode(t[n + "8"][:1].contiguous().view(torch.uint8).numpy())
                   * t[n + "d"][:1].double().numpy()[..., None, None] for n in ("q", "k", "v"))
    else:
        q, k, v = (t[n][:1].double().numpy() for n in ("q", "k", "v"))
    do = t["do"][:1].double().numpy() if w.backward else None
    bm = t["block_mask"].numpy() if "block_mask" in t else None
    nblk = max(1, w.N // REF_ROWS)

    def one(step):
        rows = np.arange((step % nblk) * REF_ROWS, min(w.N, (step % nblk + 1) * REF_ROWS))
        pairs = float(oracle.visible(w.N, w.N, w.causal, bm, rows=rows).sum())
        if w.backward:
            oracle.backward_rows(q, k, v, do, w.scale, 0, 0, rows, causal=w.causal, block_mask=bm,
                                 dropout_p=w.dropout_p, seed=w.seed)
            return pairs * 4.0 * w.d * 3.5
        oracle.forward_rows(q, k, v, w.scale, 0, 0, rows, causal=w.causal, block_mask=bm,
                            dropout_p=w.dropout_p, seed=w.seed)
        return pairs * 4.0 * w.d

    for i in range(args.warmup):
        one(i)
    flops = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops += one(i)
    total = time.perf_counter() - t0
    value = flops / total / 1e12
    sample = (f"per step: {REF_ROWS} query rows of (batch 0, head 0) of {w.B * w.H} heads, forward"
              f"{' + backward' if w.backward else ''} in fp64 with materialised score rows; steps cycle "
              f"through the head's {nblk} row blocks")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": _config(w, _density(t, w.causal)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _CORES, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- #
# the CUDA path
# --------------------------------------------------------------------------- #
def _profile_traffic(kernel_tag, workload):
    """DRAM traffic per launch from a committed ncu summary, if it was taken on
    the current source of the kernel (matching source hash); else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    src = re.search(r"source_files:\s*(.+)", text)
    if not (m and h and src):
        return None
    cur = source_sha256(src.group(1).split())
    return float(m.group(1)) if cur == h.group(1) else None


def source_sha256(files):
    """sha256 over the concatenated bytes of the given repo-relative files."""
    import hashlib
    hh = hashlib.sha256()
    for f in files:
        try:
            hh.update(open(os.path.join(ROOT, f), "rb").read())
        except OSError:
            return None
    return hh.hexdigest()


def _oracle_decode_sample(w, t, budget_s=15.0, gpu=None, parity=None):
    """Time the fp64 oracle's decode (batch, head) by (batch, head) until
    `budget_s` of oracle time has passed.  Returns (TFLOPS, seconds, heads);
    with `gpu` and `parity`, each pair's result is also compared with the
    timed step's, outside the timed calls."""
    import oracle
    heads, flops, el = 0, 0.0, 0.0
    for hh in range(w.B * w.H):
        b, h = divmod(hh, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        L = int(t["seqlens"][b])
        q, k, v = (t[n][sl].double().numpy() for n in ("q", "k", "v"))
        t0 = time.perf_counter()
        ro, rl = oracle.decode(q, k, v, w.scale, seqlens=[L], causal=w.causal)
        el += time.perf_counter() - t0
        flops += 4.0 * w.d * _decode_pairs(w.nq, L, w.causal)
        heads += 1
        if gpu is not None and parity is not None:
            parity.forward(gpu["o"][sl], gpu["lse"][sl], ro, rl)
            parity.heads += 1
        if el >= budget_s:
            break
    return flops / el / 1e12, el, heads


def _run_reference_decode(args, w):
    """Reference arm for a decode workload: each step decodes one (batch, head)
    with the fp64 oracle, cycling through the pairs."""
    import oracle
    from attn_fwd_gb300.inputs import make_decode_workload_inputs
    t = make_decode_workload_inputs(w)

    def one(step):
        hh = step % (w.B * w.H)
        b, h = divmod(hh, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        L = int(t["seqlens"][b])
        q, k, v = (t[n][sl].double().numpy() for n in ("q", "k", "v"))
        oracle.decode(q, k, v, w.scale, seqlens=[L], causal=w.causal)
        return 4.0 * w.d * _decode_pairs(w.nq, L, w.causal)

    for i in range(args.warmup):
        one(i)
    flops = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops += one(i)
    total = time.perf_counter() - t0
    value = flops / total / 1e12
    sample = (f"per step: one (batch, head) of {w.B * w.H}, {w.nq} query token(s) against its cache, fp64; "
              f"steps cycle through the pairs")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _decode_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _CORES, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _decode_config(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.nq, "N_cache": w.N, "d": w.d, "causal": w.causal,
            "cache_lengths": "uniform in [N/4, N]" if w.ragged else "full",
            "l2": "flushed (256 MiB write) between timed steps", "parallelism": "replica per GPU"}


def run_cuda_decode(args, w):
    """Decoding: fa_decode (split kernel + chunk merge) per step, the cache
    resident in HBM; roofline against the measured HBM copy bandwidth."""
    import torch
    import torch.distributed as dist

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    import attn_fwd_gb300.fa as fa
    from attn_fwd_gb300.inputs import make_decode_workload_inputs

    t = make_decode_workload_inputs(w)
    flops, nbytes = _decode_work(w, t["seqlens"].tolist())
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    sl = t["seqlens"].to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.nq), dtype=torch.float32, device=dev)
    nws = fa.fa_decode_workspace_bytes(w.B, w.H, w.nq, w.N, w.d)
    wsp = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None
    launches_per_step = 2 if nws else 1
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        fa.fa_decode(q, k, v, o, lse, sl, w.scale, causal=w.causal, workspace=wsp)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    rc = fa.fa_get_device_error()
    if rc != 0:
        raise RuntimeError(f"device status after warm-up: {fa.status_string(rc)}")
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid) if rank == 0 else None
    if sampler:
        sampler.start()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        events[i][0].record()
        step()
        events[i][1].record()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    step_ms = [e[0].elapsed_time(e[1]) for e in events]
    eager_ms = max_over_ranks(sum(step_ms), dev) / args.steps
    # the step (split kernel + chunk merge) as one CUDA-graph replay, unless --eager
    ms_per_step = eager_ms if args.eager else _graph_ms_per_step(args, step, flush, ws, dev)
    clocks = sampler.stop() if sampler else None
    rc = fa.fa_get_device_error()
    if rc != 0:
        raise RuntimeError(f"device status after timing: {fa.status_string(rc)}")
    value = whole_job_tflops(ws, flops, ms_per_step)
    timed_out = {"o": o.cpu(), "lse": lse.cpu()}

    # end to end: the new query tokens in from pinned host memory, O and LSE back
    hq = t["q"].pin_memory()
    ho, hl = torch.empty(o.shape, dtype=o.dtype).pin_memory(), torch.empty(lse.shape).pin_memory()
    e2e_steps = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(e2e_steps):
        q.copy_(hq, non_blocking=True)
        step()
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)

    peaks, peak_src = _peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = nbytes / (ms_per_step * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": "fa_decode_kernel", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": f"{peak_src} HBM copy bandwidth",
                "traffic": _profile_traffic("fa_decode_kernel", w.name),
                "algorithmic_bytes_per_step": nbytes,
                "note": "split kernel and chunk merge timed together (one step)"}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {**_decode_config(w), "launch": "eager calls" if args.eager else
                       "cuda graph of the step, one replay per step"},
            "eager_ms_per_step": eager_ms,
            "e2e": {"value": whole_job_tflops(ws, flops, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": hq.numel() * hq.element_size(),
                    "d2h_bytes_per_step": ho.numel() * ho.element_size() + hl.numel() * hl.element_size(),
                    "ms_per_step": e2e_ms},
            "gpu_launches": launches_per_step * args.steps, "roofline": roofline, "clocks": clocks}
    rc_out = 0
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        par = Parity()
        tf, el, heads = _oracle_decode_sample(w, t, budget_s=args.cpu_budget, gpu=timed_out, parity=par)
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": _CORES, "kind": "oracle",
                                "sample": f"{heads} of {w.B * w.H} (batch, head) pairs, decode, fp64, {el:.1f} s"}
        line["parity"] = par.report(False)
        rc_out = 0 if line["parity"]["ok"] else 1
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return rc_out


def _run_cuda_fp8(args, w, t, f_fwd, fa, dev, ws, rank):
    """8-bit forward: fa_fwd_fp8 (V transpose + forward kernel) per step;
    roofline against the 8-bit tensor peak = measured bf16 peak x 2 (the
    nominal dense fp8 : bf16 ratio, 4.5 : 2.25 PFLOP/s)."""
    import torch
    import torch.distributed as dist
    d8 = {n: t[n].to(dev) for n in ("q8", "k8", "v8", "qd", "kd", "vd")}
    o = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    wsp = torch.empty(fa.fa_fwd_fp8_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        fa.fa_fwd_fp8(d8["q8"], d8["k8"], d8["v8"], o, lse, d8["qd"], d8["kd"], d8["vd"], w.scale, w.causal, wsp)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if fa.fa_get_device_error() != 0:
        raise RuntimeError("device status after warm-up")
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid) if rank == 0 else None
    if sampler:
        sampler.start()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        events[i][0].record()
        step()
        events[i][1].record()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    eager_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in events), dev) / args.steps
    # the step (V transpose + forward) as one CUDA-graph replay, unless --eager
    ms_per_step = eager_ms if args.eager else _graph_ms_per_step(args, step, flush, ws, dev)
    clocks = sampler.stop() if sampler else None
    if fa.fa_get_device_error() != 0:
        raise RuntimeError("device status after timing")
    value = whole_job_tflops(ws, f_fwd, ms_per_step)
    timed_out = {"o": o.cpu(), "lse": lse.cpu()}
    host_in = {n: t[n].pin_memory() for n in d8}
    ho, hl = torch.empty(o.shape, dtype=o.dtype).pin_memory(), torch.empty(lse.shape).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(e2e_steps):
        for n, x in host_in.items():
            d8[n].copy_(x, non_blocking=True)
        step()
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    peaks, peak_src = _peaks()
    peak = 2.0 * float(peaks["bf16_tflops"])
    achieved = f_fwd / (ms_per_step * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": "fa_fwd_fp8_kernel", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{peak_src} bf16 dense (burst) x 2, the nominal e4m3 : bf16 ratio",
                "traffic": _profile_traffic("fa_fwd_fp8_kernel", w.name), "algorithmic_flops_per_launch": f_fwd,
                "note": "timed with the V transpose launch that precedes it"}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3", "data": "synthetic", "config": {**_config(w, None), "inputs":
            f"N(0,1) seed {w.seed}, e4m3 with per-(batch, head) descale amax/448",
            "launch": "eager calls" if args.eager else "cuda graph of the step, one replay per step"},
            "eager_ms_per_step": eager_ms,
            "e2e": {"value": whole_job_tflops(ws, f_fwd, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in host_in.values()),
                    "d2h_bytes_per_step": ho.numel() * ho.element_size() + hl.numel() * hl.element_size(),
                    "ms_per_step": e2e_ms},
            "gpu_launches": 2 * args.steps, "roofline": roofline, "clocks": clocks}
    rc_out = 0
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        par = Parity()
        tf, el, heads = _oracle_sample(w, t, budget_s=args.cpu_budget, gpu=timed_out, parity=par)
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": _CORES, "kind": "oracle",
                                "sample": f"{heads} of {w.B * w.H} (batch, head) pairs, 8-bit forward, fp64, {el:.1f} s"}
        line["parity"] = par.report(False)
        rc_out = 0 if line["parity"]["ok"] else 1
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return rc_out


def _read(path):
    try:
        with open(path) as f:
            return f.read().strip()
    except OSError:
        return None


def _host_link_info(dev):
    """Where the host side of the end-to-end copies sits (read-only: sysfs and
    the process status), and the pinned copy rates, each direction alone, on
    256 MiB buffers timed with CUDA events (outside any timed step)."""
    import torch
    info = {}
    try:
        p = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        info["gpu_pci"] = bus
        info["gpu_numa_node"] = _read(f"/sys/bus/pci/devices/{bus}/numa_node")
        info["gpu_local_cpus"] = _read(f"/sys/bus/pci/devices/{bus}/local_cpulist")
    except Exception:
        pass
    nodes = _read("/sys/devices/system/node/online")
    info["numa_nodes_online"] = nodes
    if hasattr(os, "sched_getaffinity"):
        cpus = sorted(os.sched_getaffinity(0))
        info["process_cpus"] = f"{cpus[0]}-{cpus[-1]}" if cpus == list(range(cpus[0], cpus[-1] + 1)) else cpus
    status = _read("/proc/self/status") or ""
    for line in status.splitlines():
        if line.startswith("Mems_allowed_list"):
            info["pinned_memory_nodes_allowed"] = line.split(":", 1)[1].strip()
    try:
        n = 256 << 20
        h = torch.empty(n, dtype=torch.uint8).pin_memory()
        d = torch.empty(n, dtype=torch.uint8, device=dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for direction in ("h2d", "d2h"):
            best = None
            for _ in range(3):
                torch.cuda.synchronize()
                e0.record()
                (d.copy_(h, non_blocking=True) if direction == "h2d" else h.copy_(d, non_blocking=True))
                e1.record()
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1)
                best = ms if best is None else min(best, ms)
            info[f"{direction}_gbs"] = n / (best * 1e-3) / 1e9
        del h, d
    except Exception:
        pass
    return info


def _graph_ms_per_step(args, step, flush, ws, dev):
    """Capture step() into a CUDA graph and time one replay per step (CUDA
    events around each replay, the L2 flushed before each, max over ranks)."""
    import torch
    import torch.distributed as dist
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(args.warmup):
        flush.zero_()
        g.replay()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for ev in events:
        flush.zero_()
        ev[0].record()
        g.replay()
        ev[1].record()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    total = sum(e0.elapsed_time(e1) for e0, e1 in events)
    return max_over_ranks(total, dev) / args.steps


def run_cuda(args):
    import torch
    import torch.distributed as dist
    from attn_fwd_gb300.inputs import DECODE_WORKLOADS
    if args.workload in DECODE_WORKLOADS:
        return run_cuda_decode(args, DECODE_WORKLOADS[args.workload])

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import attn_fwd_gb300.fa as fa
    from attn_fwd_gb300.inputs import WORKLOADS, make_workload_inputs

    w = WORKLOADS[args.workload]
    t = make_workload_inputs(w)
    density = _density(t, w.causal)
    f_fwd, f_bwd = _flops(w, density)
    if w.fp8:
        return _run_cuda_fp8(args, w, t, f_fwd, fa, dev, ws, rank)
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    do = t["do"].to(dev) if w.backward else None
    bm = t["block_mask"].to(dev) if "block_mask" in t else None
    mask_kind = (fa.MASK_BLOCK if bm is not None else 0) | (fa.MASK_CAUSAL if w.causal else 0)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    if w.backward:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        wsp = fa.workspace(w.B, w.H, w.N, w.d, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def fwd():
        if w.dropout_p:
            fa.fa_fwd_dropout(q, k, v, o, lse, bm, w.scale, w.causal, w.dropout_p, w.seed)
        elif bm is not None:
            fa.fa_fwd_blocksparse(q, k, v, o, lse, bm, w.scale, causal=w.causal)
        else:
            fa.fa_fwd(q, k, v, o, lse, w.scale, causal=w.causal)

    def step(ev=None):
        if ev:
            ev[0].record()
        fwd()
        if ev:
            ev[1].record()
        if w.backward:
            fa.fa_bwd_preprocess(o, do, lse, wsp)
            if ev:
                ev[2].record()
            fa.fa_bwd_main(q, k, v, do, bm, dk, dv, wsp, w.scale, mask_kind, w.dropout_p, w.seed)
            if ev:
                ev[3].record()
            fa.fa_bwd_dq_convert(wsp, dq, w.scale)
            if ev:
                ev[4].record()

    launches_per_step = 4 if w.backward else 1
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    rc = fa.fa_get_device_error()
    if rc != 0:
        raise RuntimeError(f"device status after warm-up: {fa.status_string(rc)}")

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid) if rank == 0 else None
    if sampler:
        sampler.start()
    nev = 5 if w.backward else 2
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        step(events[i])
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    rc = fa.fa_get_device_error()
    if rc != 0:
        raise RuntimeError(f"device status after timing: {fa.status_string(rc)}")

    per = {"fwd": [], "bwd_preprocess": [], "bwd_main": [], "bwd_dq_convert": []}
    step_ms = []
    for ev in events:
        step_ms.append(ev[0].elapsed_time(ev[-1]))
        per["fwd"].append(ev[0].elapsed_time(ev[1]))
        if w.backward:
            per["bwd_preprocess"].append(ev[1].elapsed_time(ev[2]))
            per["bwd_main"].append(ev[2].elapsed_time(ev[3]))
            per["bwd_dq_convert"].append(ev[3].elapsed_time(ev[4]))
    total_ms = max_over_ranks(sum(step_ms), dev)
    ms_per_step = total_ms / args.steps
    eager_ms_per_step = ms_per_step
    if not args.eager:
        # the same step captured once and replayed: no host work between the
        # kernels, which is what bounds one-tile and other launch-bound shapes
        ms_per_step = _graph_ms_per_step(args, step, flush, ws, dev)
        rc = fa.fa_get_device_error()
        if rc != 0:
            raise RuntimeError(f"device status after the graph replays: {fa.status_string(rc)}")
    clocks = sampler.stop() if sampler else None
    value = whole_job_tflops(ws, f_fwd + f_bwd, ms_per_step)
    # the outputs of the last timed step, for the parity check against the oracle
    timed_out = {"o": o.cpu(), "lse": lse.cpu()}
    if w.backward:
        timed_out.update({"dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu()})

    # ---- end to end through the public binding, host buffers ------------- #
    host_in = {n: t[n].pin_memory() for n in (("q", "k", "v", "do") if w.backward else ("q", "k", "v"))}
    host_out = {"o": torch.empty(q.shape, dtype=q.dtype).pin_memory(),
                "lse": torch.empty(lse.shape, dtype=lse.dtype).pin_memory()}
    if w.backward:
        for n in ("dq", "dk", "dv"):
            host_out[n] = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in host_out.values())
    dev_in = {"q": q, "k": k, "v": v}
    if w.backward:
        dev_in["do"] = do
    dev_out = {"o": o, "lse": lse}
    if w.backward:
        dev_out.update({"dq": dq, "dk": dk, "dv": dv})
    e2e_steps = max(3, min(args.steps, 20))
    # forward + backward without dropout: the library's host-streamed entry
    # point (copies in, kernels and copies out of successive chunks of heads
    # overlap); otherwise pinned copies around the device-resident step
    streamed = not w.dropout_p
    if streamed and w.backward:
        hws = torch.empty(fa.fa_fwd_bwd_host_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)

        def e2e_step():
            fa.fa_fwd_bwd_host(host_in["q"], host_in["k"], host_in["v"], host_in["do"], host_out["o"],
                               host_out["lse"], host_out["dq"], host_out["dk"], host_out["dv"], bm, hws, w.scale,
                               w.causal)
    elif streamed:
        hws = torch.empty(fa.fa_fwd_host_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)

        def e2e_step():
            fa.fa_fwd_host(host_in["q"], host_in["k"], host_in["v"], host_out["o"], host_out["lse"], bm, hws,
                           w.scale, w.causal)
    else:
        def e2e_step():
            for n, x in host_in.items():
                dev_in[n].copy_(x, non_blocking=True)
            step()
            for n, x in dev_out.items():
                host_out[n].copy_(x, non_blocking=True)
    e2e_step()                                  # warm-up (streams, tensor maps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(e2e_steps):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    e2e_value = whole_job_tflops(ws, f_fwd + f_bwd, e2e_ms)
    # what the end-to-end call returned against the timed device step's outputs
    e2e_diff = {n: float((host_out[n].float() - timed_out[n].float()).abs().max()) for n in host_out}

    # ---- roofline of the dominant kernel -------------------------------- #
    peaks, peak_src = _peaks()
    avg = {kname: (sum(x) / len(x) if x else 0.0) for kname, x in per.items()}
    algo = {"fwd": f_fwd, "bwd_main": f_bwd}
    dom = max(("fwd", "bwd_main") if w.backward else ("fwd",), key=lambda n: avg[n])
    achieved = algo[dom] / (avg[dom] * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    tag = {"fwd": "fa_fwd_kernel", "bwd_main": "fa_bwd_kernel"}[dom]
    roofline = {"bound": "tensor", "kernel": tag, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": f"{peak_src} bf16 dense (burst)",
                "traffic": _profile_traffic(tag, w.name),
                "algorithmic_flops_per_launch": algo[dom],
                "other_peaks": _other_peaks(achieved, peaks, clocks, dev)}
    kernels = {kname: {"ms": avg[kname], "share": avg[kname] / eager_ms_per_step if eager_ms_per_step else 0.0}
               for kname in avg if per[kname]}
    kernels["fwd"]["tflops"] = f_fwd / (avg["fwd"] * 1e-3) / 1e12
    kernels["fwd"]["frac_of_peak"] = kernels["fwd"]["tflops"] / peak
    if w.backward:
        kernels["bwd_main"]["tflops"] = f_bwd / (avg["bwd_main"] * 1e-3) / 1e12
        kernels["bwd_main"]["frac_of_peak"] = kernels["bwd_main"]["tflops"] / peak
        bwd_ms = avg["bwd_preprocess"] + avg["bwd_main"] + avg["bwd_dq_convert"]
        kernels["bwd_total"] = {"ms": bwd_ms, "tflops": f_bwd / (bwd_ms * 1e-3) / 1e12,
                                "frac_of_peak": f_bwd / (bwd_ms * 1e-3) / 1e12 / peak}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": _config(w, density, {"launch": "eager calls" if args.eager else
                                           "cuda graph of the step, one replay per step"}),
            "frac_of_peak": value / ws / peak,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms,
                    "call": ((("fa_fwd_bwd_host" if w.backward else "fa_fwd_host") +
                              ": chunks of heads, copies overlapped with the kernels") if streamed
                             else "pinned copies in, device-resident step, copies out"),
                    "max_abs_diff_vs_device_step": e2e_diff,
                    "host_link": _host_link_info(dev)},
            "gpu_launches": launches_per_step * args.steps, "roofline": roofline, "kernels": kernels,
            "clocks": clocks}
    if not args.eager:
        line["eager_ms_per_step"] = eager_ms_per_step

    rc_out = 0
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        par = Parity()
        tf, el, heads = _oracle_sample(w, t, budget_s=args.cpu_budget, gpu=timed_out, parity=par)
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": _CORES, "kind": "oracle",
                                "sample": f"{heads} of {w.B * w.H} (batch, head) pairs, forward"
                                          f"{' + backward' if w.backward else ''}, fp64, {el:.1f} s"}
        line["parity"] = par.report(w.backward)
        rc_out = 0 if line["parity"]["ok"] else 1
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return rc_out


def _apply_overrides(args, ap):
    """--set K=V,...: a copy of the workload with some sizes replaced, under
    the name '<workload>@<overrides>' (no stored profile matches it)."""
    import dataclasses
    from attn_fwd_gb300.inputs import DECODE_WORKLOADS, WORKLOADS
    table = DECODE_WORKLOADS if args.workload in DECODE_WORKLOADS else WORKLOADS
    if args.workload not in table:
        ap.error(f"unknown workload {args.workload}")
    w = table[args.workload]
    kw = {}
    for item in args.set.split(","):
        key, _, val = item.partition("=")
        if not hasattr(w, key) or key in ("name", "note"):
            ap.error(f"--set: unknown field {key}")
        cur = getattr(w, key)
        kw[key] = (val.lower() in ("1", "true", "yes")) if isinstance(cur, bool) else type(cur)(val) \
            if cur is not None else float(val)
    name = f"{w.name}@{args.set}"
    table[name] = dataclasses.replace(w, name=name, **kw)
    args.workload = name


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=("cuda", "reference"), default="cuda")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="time the step as eager calls instead of one replay of a CUDA graph of the step "
                         "(per-kernel times and the roofline are always taken from eager calls)")
    ap.add_argument("--set", default="", metavar="K=V,...",
                    help="override sizes of the workload, e.g. N=2048,H=16 (an ad-hoc shape with its recipe)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.set:
        _apply_overrides(args, ap)
    if args.impl == "reference":
        return run_reference(args)
    return run_cuda(args)


if __name__ == "__main__":
    sys.exit(main())
