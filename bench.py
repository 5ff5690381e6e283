"""Benchmark of the packed document-causal attention hot path on one GB300.

One step is the whole path over one batch of synthetic input already resident
in HBM. On the default workload (65536 packed tokens, document lengths
Pareto(1.2) in [256, 32768], tail padded, Hq=32, Hkv=8, D=128, bf16, scale
1/sqrt(128)) a step is:

  (i)  document-causal attention of the whole row with a left window of 4096:
       doc-ids -> segment builder (padding runs as key-less query segments, so
       the forward itself writes the padding rows' zero output and -inf lse),
       forward (schedule, uncovered-row fill, attention) and backward
       (schedule, Delta preprocess, attention backward, dQ/dK/dV convert);
  (ii) the cross-chunk run without window of the query shard 32768..65535:
       its local key chunk (keys 32768..65535, document-causal through the
       builder) and its cross chunk (keys 0..32767, non-causal through the
       cross-chunk builder), the cross result merged into the local one by
       lse on its live rows, both chunks' backward from the merged out/lse,
       and the cross chunk's dQ added on its live rows.

Metric: forward + backward TFLOP/s counting only unmasked work (pad queries and
zero-query segments excluded): forward 2 (Dqk + Dv) and backward
(6 Dqk + 4 Dv) flops per visible (query, key) pair per query head.

  python bench.py [--gpus N --steps K --warmup W]      our CUDA path
  python bench.py --impl reference ...                  the fp64 CPU oracle
  python bench.py --config 2|3|4|6                      the other workloads

Under torchrun (N > 1) every rank runs its own replica on its own GPU (no
collective on the data path; weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from packed_sequence_flash_gb300 import inputs  # noqa: E402

METRIC = "varlen doc-causal attention fwd/bwd TFLOP/s (bf16) and % of GB300 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
# CPU legs: the oracle's work per timed sample (about 15 s on 16 host cores for
# the cpu_baseline, about 5 s per step for the reference arm)
CPU_SAMPLE_GFLOP = 300.0
REF_STEP_GFLOP = 100.0
# The reference arm's whole run (warm-up + timed steps) is held to about this
# much oracle work, a couple of minutes on the host cores, by shrinking each
# step's sample when many steps are asked for.
REF_TOTAL_GFLOP = 2000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
# dram__bytes_read.sum + dram__bytes_write.sum of a main kernel per step (the
# sum over the step's launches of it) from one ncu capture: (kernel, workload)
# -> (hash of the kernel's sources when captured, bytes). Reported as null for
# other workloads and once the sources change.
NCU_TRAFFIC = {
    # the document path's default: a KV head's query heads packed into one tile
    ("attn_fwd_duo_kernel", "cfg5_doc_causal_t65536_w4096"): ("88fbcdf5a2921253", 3777393920),
    ("attn_bwd_dual_kernel", "cfg5_doc_causal_t65536_w4096"): ("3ecea61619644db9", 35805310720),
    ("attn_fwd_duo_kernel", "cfg2_doc_causal_t8192_d128"): ("88fbcdf5a2921253", 52276992),
    ("attn_bwd_dual_kernel", "cfg2_doc_causal_t8192_d128"): ("3ecea61619644db9", 362997760),
    ("attn_fwd_pair_kernel", "cfg4_doc_causal_shard_dqk192_dv128"): ("5837d1098189c960", 185433856),
    ("attn_bwd_kernel", "cfg4_doc_causal_shard_dqk192_dv128"): ("26951fb59a1df2f0", 775970048),
    ("attn_fwd_kernel", "cfg3_dense_causal_n4096_d512"): ("cf0774645e2e7eda", 126322944),
    ("attn_bwd_wide_kernel", "cfg3_dense_causal_n4096_d512"): ("df0f829a9fa47815", 960428544),
}


def ncu_traffic(kernel: str, workload: str):
    """Captured DRAM bytes per launch of `kernel` on `workload`, or None."""
    cap = NCU_TRAFFIC.get((kernel, workload))
    return cap[1] if cap and cap[0] == kernel_source_hash(kernel) else None

# Sources each main kernel is compiled from (for the hash above).
KERNEL_SOURCES = {
    "attn_fwd_duo_kernel": ("fwd.cuh", "fwd_duo.cuh", "common.cuh", "ptx.cuh"),
    "attn_fwd_kernel": ("fwd.cuh", "fwd512.cuh", "common.cuh", "ptx.cuh"),
    "attn_fwd_pair_kernel": ("fwd.cuh", "fwd_pair.cuh", "common.cuh", "ptx.cuh"),
    "attn_bwd_dual_kernel": ("bwd.cuh", "bwd_dual.cuh", "common.cuh", "ptx.cuh"),
    "attn_bwd_kernel": ("bwd.cuh", "bwd192.cuh", "common.cuh", "ptx.cuh"),
    "attn_bwd_wide_kernel": ("bwd.cuh", "bwd_wide.cuh", "cluster.cuh", "common.cuh", "ptx.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "packed_sequence_flash_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def main_kernels(dqk: int, dv: int) -> tuple[str, str]:
    """Names of the forward and backward kernels the library runs for these head dims."""
    if dqk == dv and dqk in (64, 128):
        fwd = "attn_fwd_duo_kernel"
    elif (dqk, dv) == (192, 128):
        fwd = "attn_fwd_pair_kernel"
    else:
        fwd = "attn_fwd_kernel"
    if dqk <= 128 and dv <= 128:
        bwd = "attn_bwd_dual_kernel"
    elif dqk == 512 and dv == 512:
        bwd = "attn_bwd_wide_kernel"
    else:
        bwd = "attn_bwd_kernel"
    return fwd, bwd


def visible_pairs(doc_ids: np.ndarray, q0: int, Lq: int, window=None) -> int:
    """Pairs (query, key) a non-padding query of the shard sees, summed over rows."""
    total = 0
    for row in np.asarray(doc_ids):
        S = row.shape[0]
        change = np.ones(S, bool)
        change[1:] = row[1:] != row[:-1]
        run_start = np.maximum.accumulate(np.where(change, np.arange(S), 0))
        p = np.arange(q0, q0 + Lq)
        cnt = p - run_start[p] + 1
        if window:
            cnt = np.minimum(cnt, window)
        total += int(cnt[row[p] != 0].sum())
    return total


def dense_pairs(Nq: int, Nk: int, causal: bool) -> int:
    """Visible pairs of one dense [Nq x Nk] problem (causal: bottom-right aligned)."""
    if not causal:
        return Nq * Nk
    return sum(max(0, min(Nk, i + Nk - Nq + 1)) for i in range(Nq))


def workload_flops(w):
    """(visible pairs x query heads, forward flops, backward flops) of one step."""
    if w.kind == "dense":
        B, Hq, Nq, Dqk = w.q.shape
        Nk, Dv = w.k.shape[2], w.v.shape[3]
        pairs = B * Hq * dense_pairs(Nq, Nk, w.causal)
    else:
        Lq = w.q.shape[0]
        Hq, Dqk, Dv = w.q.shape[1], w.q.shape[2], w.v.shape[2]
        pairs = visible_pairs(w.doc_ids, w.q_global_start, Lq, w.window) * Hq
        split = w.extra.get("cross_split")
        if split:
            # the cross-chunk run: the shard's queries against both chunks, no
            # window (local + cross pairs = the unsplit shard's pairs)
            pairs += visible_pairs(w.doc_ids, split, w.k.shape[0] - split, None) * Hq
    return pairs, pairs * 2 * (Dqk + Dv), pairs * (6 * Dqk + 4 * Dv)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as fh:
                return json.load(fh), "measured"
        except Exception:
            pass
    return {}, "fallback"


class ClockSampler:
    """nvidia-smi samples every 100 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self):
        return time.time()

    def summary(self, t0, t1):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [r for t, r in self.rows if t0 - 0.1 <= t <= t1 + 0.25] or [r for _, r in self.rows[-3:]]
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def doc_pairs(n: int, window=None) -> int:
    """Visible pairs of one causal document of n tokens (left window counting the current token)."""
    if not window or window >= n:
        return n * (n + 1) // 2
    return window * (window + 1) // 2 + (n - window) * window


def cpu_sample_workload(w, gflop, offset_docs=0):
    """Whole documents from offset_docs on, about `gflop` GFLOP of forward +
    backward work (at least one document), as a workload of its own (same
    distribution, same window, exact flops)."""
    lengths = w.extra["lengths"]
    Hq, Dqk, Dv = w.q.shape[1], w.q.shape[2], w.v.shape[2]
    per_pair = Hq * (2 * (Dqk + Dv) + 6 * Dqk + 4 * Dv)
    budget = gflop * 1e9
    pos = sum(lengths[:offset_docs])
    start = pos
    flops = 0.0
    i = offset_docs
    taken = []
    while i < len(lengths) and (i == offset_docs or flops + doc_pairs(lengths[i], w.window) * per_pair <= budget):
        n = lengths[i]
        if i == offset_docs and doc_pairs(n, w.window) * per_pair > budget:
            # a first document alone over budget: its leading tokens (a causal
            # document of its own) up to the budget
            n = 1
            while n < lengths[i] and doc_pairs(2 * n, w.window) * per_pair <= budget:
                n *= 2
        flops += doc_pairs(n, w.window) * per_pair
        pos += n
        taken.append(n)
        i += 1
        if n < lengths[i - 1]:
            break
    name = f"{w.name}[docs {offset_docs}..{i - 1}" + ("" if taken[-1] == lengths[i - 1] else
                                                       f", the first {taken[-1]} tokens of the last") + "]"
    sub = inputs.Workload(name, "document", w.q[start:pos], w.k[start:pos], w.v[start:pos], w.dout[start:pos],
                          w.scale, True, w.window, w.doc_ids[:, start:pos] - w.doc_ids[0, start] + 1, 0)
    sub.extra["lengths"] = taken
    return sub, i - offset_docs


def cpu_sample_dense(w, n_max=1024):
    """Batch 0, the first KV head and its query heads, the leading n x n block
    (itself a causal problem when Nq = Nk)."""
    B, Hq, Nq, _ = w.q.shape
    Hkv, Nk = w.k.shape[1], w.k.shape[2]
    G = Hq // Hkv
    n = min(Nq, Nk, n_max)
    sub = inputs.Workload(f"{w.name}[b0, kv head 0, {n} rows]", "dense", w.q[:1, :G, :n], w.k[:1, :1, :n],
                          w.v[:1, :1, :n], w.dout[:1, :G, :n], w.scale, w.causal)
    return sub


def run_oracle(sub, nthreads, softcap=None):
    import oracle

    t = time.perf_counter()
    if sub.kind == "dense":
        out, lse = oracle.attn_fwd_dense(sub.q, sub.k, sub.v, sub.scale, sub.causal, nthreads=nthreads,
                                         softcap=softcap)
        oracle.attn_bwd_dense(sub.dout, sub.q, sub.k, sub.v, out, lse, sub.scale, sub.causal, nthreads=nthreads,
                              softcap=softcap)
        return time.perf_counter() - t
    out, lse = oracle.attn_fwd_document(sub.q, sub.k, sub.v, sub.doc_ids, 0, sub.scale, sub.window,
                                        nthreads=nthreads, softcap=softcap)
    oracle.attn_bwd_document(sub.dout, sub.q, sub.k, sub.v, out, lse, sub.doc_ids, 0, sub.scale, sub.window,
                             nthreads=nthreads, softcap=softcap)
    return time.perf_counter() - t


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, softcap=None):
    if w.kind == "dense":
        sub = cpu_sample_dense(w)
        what = f"{sub.name}"
    else:
        sub, ndocs = cpu_sample_workload(w, CPU_SAMPLE_GFLOP)
        what = (f"the first {ndocs} of {len(w.extra['lengths'])} documents of the row ({sub.q.shape[0]} tokens"
                + (f", window {w.window}" if w.window else ""))
    _, f, b = workload_flops(sub)
    c = cores()
    secs = run_oracle(sub, c, softcap)
    what = what + (")" if w.kind != "dense" else "")
    return {"value": (f + b) / secs / 1e12, "unit": UNIT, "cores": c, "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd on {what}, {(f + b) / 1e9:.1f} GFLOP, once, {secs:.1f} s"}


def config_dict(w, args, pairs, n_docs, world=1):
    """The workload's description; both arms print the same keys."""
    common = {"visible_pairs_x_heads": int(pairs), "seed": args.seed, "l2": "flushed between steps (256 MiB write)",
              "pack_gqa": bool(getattr(args, "pack_gqa", False)), "softcap": getattr(args, "softcap", None),
              "parallelism": f"replicas{world}" if world > 1 else "single GPU"}
    if w.kind == "dense":
        B, Hq, Nq, Dqk = w.q.shape
        return dict({"workload": w.name, "batch": int(B), "q_rows": int(Nq), "k_rows": int(w.k.shape[2]),
                     "Hq": int(Hq), "Hkv": int(w.k.shape[1]), "Dqk": int(Dqk), "Dv": int(w.v.shape[3]),
                     "causal": bool(w.causal)}, **common)
    d = {"workload": w.name, "tokens": int(w.k.shape[0]), "q_tokens": int(w.q.shape[0]),
         "q_global_start": int(w.q_global_start), "Hq": int(w.q.shape[1]), "Hkv": int(w.k.shape[1]),
         "Dqk": int(w.q.shape[2]), "Dv": int(w.v.shape[2]), "window": w.window, "documents": n_docs}
    split = w.extra.get("cross_split")
    if split:
        d["cross_chunk_run"] = (f"queries {split}..{w.k.shape[0] - 1} without window: local chunk keys "
                                f"{split}..{w.k.shape[0] - 1} (causal) + cross chunk keys 0..{split - 1} "
                                "(non-causal), merged by lse")
    return dict(d, **common)


# ---------------------------------------------------------------------------

# ---------------------------------------------------------------------------
# ranks: one replica per GPU, no collective on the data path

def replica_seed(seed: int, rank: int) -> int:
    """Each rank runs its own replica of the workload, drawn with its own seed."""
    return seed + rank


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The largest of the ranks' values, on every rank (the timing rule: a
    step takes as long as the slowest replica)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def roofline_peak(peaks: dict, src: str, ms_per_step: float, steps: int):
    """(peak, burst peak, description) in TFLOP/s for the main kernels' roofline.

    The kernels are timed inside the step: for a long step (10 ms or more,
    back-to-back launches under the power cap) or a timed loop of seconds the
    sustained peak is the denominator, else the burst peak; the caller reports
    the fraction of the burst peak as well."""
    measured = src == "measured"
    burst = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS)) if measured else FALLBACK_BF16_TFLOPS
    sustained = (float(peaks.get("bf16_tflops_sustained", FALLBACK_BF16_TFLOPS_SUSTAINED)) if measured
                 else FALLBACK_BF16_TFLOPS_SUSTAINED)
    long_loop = ms_per_step >= 10.0 or steps * ms_per_step >= 1000.0
    kind = "bf16 dense sustained (kernels timed inside a long step)" if long_loop else "bf16 dense burst"
    return (sustained if long_loop else burst), burst, f"{kind}, {'of measured' if measured else 'of fallback'}"


def whole_job_value(world: int, flops_per_replica: float, ms_max: float) -> float:
    """Whole-job TFLOP/s: every replica's work over the slowest replica's time."""
    return world * flops_per_replica / (ms_max * 1e-3) / 1e12


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:  # the oracle runs once, on rank 0; other ranks exit without work
        return 0
    w = inputs.config(args.config, args.seed)
    pairs, _, _ = workload_flops(w)
    c = cores()
    total_f, total_s = 0.0, 0.0
    per = []
    dense = w.kind == "dense"
    ndocs_total = 0 if dense else len(w.extra["lengths"])
    step_gflop = min(REF_STEP_GFLOP, REF_TOTAL_GFLOP / max(args.warmup + args.steps, 1))
    for s in range(args.warmup + args.steps):
        if dense:
            sub = cpu_sample_dense(w, 512)
        else:
            sub, nd = cpu_sample_workload(w, step_gflop, offset_docs=s % max(ndocs_total - 1, 1))
        _, f, b = workload_flops(sub)
        secs = run_oracle(sub, c, args.softcap)
        if s >= args.warmup:
            total_f += f + b
            total_s += secs
            per.append(secs)
    value = total_f / total_s / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": config_dict(w, args, pairs, ndocs_total, int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": c, "kind": "oracle",
                             "sample": (f"each step: fp64 oracle fwd+bwd on {sub.name} (batch 0, the first KV "
                                        "head and its query heads, the leading causal block)" if dense else
                                        "each step: fp64 oracle fwd+bwd on a run of whole documents (same "
                                        f"window) of about {step_gflop:.1f} GFLOP (at least one document, the "
                                        "leading tokens of one when a whole one is larger), starting one "
                                        "document later each step")},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line))
    return 0


def our_arm(args):
    import torch

    import packed_sequence_flash_gb300 as psf
    from packed_sequence_flash_gb300 import _lib

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    lib = _lib.load()

    w = inputs.config(args.config, replica_seed(args.seed, rank))
    if args.dtype == "fp16":
        # the same draws held as fp16 (fp16 storage and fp16 tensor-core inputs)
        w.q, w.k, w.v, w.dout = (t.to(torch.float16) for t in (w.q, w.k, w.v, w.dout))
    pairs, f_fwd, f_bwd = workload_flops(w)
    flops = f_fwd + f_bwd
    Lq = w.q.shape[0]
    q, k, v, do = (t.to(dev) for t in (w.q, w.k, w.v, w.dout))
    dense = w.kind == "dense"
    if dense:
        ids = qids = None
    else:
        ids = torch.from_numpy(np.ascontiguousarray(w.doc_ids)).to(dev)
        qids = ids[:, w.q_global_start:w.q_global_start + Lq].contiguous()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    split = None if dense else w.extra.get("cross_split")

    def cross_chunk_run(qq, kk, vv, dd, ii):
        """The shard [split, S) without window: local chunk (causal, through the
        builder) and cross chunk (non-causal, through the cross-chunk builder),
        merged by lse on the cross chunk's live rows; both backwards from the
        merged out/lse; the cross dQ added on its live rows."""
        S = kk.shape[0]
        qs, ds = qq[split:], dd[split:]
        kl, vl, kc, vc = kk[split:], vv[split:], kk[:split], vv[:split]
        ids_l = ii[:, split:]
        out, lse, seg = psf.document_causal_attention(qs, kl, vl, ids_l, ids_l, 0, w.scale, softcap=args.softcap,
                                                      pack_gqa=args.pack_gqa)
        cq, ck, meta = psf.build_cross_segments(ii, split, S - split, 0, split)
        out_c, lse_c = psf.attn_varlen_fwd(qs, kc, vc, cq, ck, -1, -1, w.scale, False, dev_meta=meta,
                                           softcap=args.softcap, pack_gqa=args.pack_gqa)
        psf.lse_merge_live_rows(out, lse, out_c, lse_c, cq, ck, dev_meta=meta)
        dq, dkl, dvl = psf.document_causal_attention_backward(ds, qs, kl, vl, out, lse, seg, w.scale,
                                                              softcap=args.softcap, pack_gqa=args.pack_gqa)
        dqc, dkc, dvc = psf.attn_varlen_bwd(ds, qs, kc, vc, out, lse, cq, ck, -1, -1, w.scale, False,
                                            dev_meta=meta, softcap=args.softcap, pack_gqa=args.pack_gqa)
        psf.grad_add_live_rows(dq, dqc, cq, ck, dev_meta=meta)
        return out, lse, (dq, dkc, dkl, dvc, dvl)

    def step(qq, kk, vv, dd, ii, qi):
        if dense:
            out, lse = psf.attn_dense_fwd(qq, kk, vv, w.scale, w.causal, pack_gqa=args.pack_gqa,
                                          softcap=args.softcap)
            grads = psf.attn_dense_bwd(dd, qq, kk, vv, out, lse, w.scale, w.causal, softcap=args.softcap,
                                       pack_gqa=args.pack_gqa)
            return (out, lse) + tuple(grads)
        out, lse, seg = psf.document_causal_attention(qq, kk, vv, qi, ii, w.q_global_start, w.scale, w.window,
                                                      pack_gqa=args.pack_gqa, softcap=args.softcap)
        grads = psf.document_causal_attention_backward(dd, qq, kk, vv, out, lse, seg, w.scale, w.window,
                                                       softcap=args.softcap, pack_gqa=args.pack_gqa)
        res = (out, lse) + tuple(grads)
        if split:
            o2, l2, g2 = cross_chunk_run(qq, kk, vv, dd, ii)
            res += (o2, l2) + g2
        return res

    for _ in range(args.warmup):
        step(q, k, v, do, ids, qids)
    torch.cuda.synchronize()
    if psf.device_status() != 0:
        raise RuntimeError("device status after warm-up is not OK")

    # ---- eager steps: per-step time and the main kernels' own launch times
    def timed(run_one, n):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        stops = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            flush.zero_()
            starts[i].record()
            run_one()
            stops[i].record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(starts, stops)]

    def kernel_times():
        """{"fwd"/"bwd": (summed ms, launches)} of the recorded main-kernel events."""
        kt = {}
        for kind, name in ((0, "fwd"), (1, "bwd")):
            tot = ctypes_double()
            n = ctypes_int()
            _lib.check(lib.psf_kernel_times_ms(kind, tot, n))
            kt[name] = (tot.value, n.value)
        return kt

    run_step = lambda: step(q, k, v, do, ids, qids)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    lib.psf_kernel_timing(1)
    eager_steps = timed(run_step, args.steps)
    lib.psf_kernel_timing(0)
    kt_eager = kernel_times()
    if psf.device_status() != 0:
        raise RuntimeError("device status after the eager steps is not OK")

    # ---- the step replayed as one CUDA graph (same kernels, no launch gaps)
    graph, graph_note = None, None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            run_step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        # the main kernels' event pairs become nodes of the graph: every replay
        # re-records them, so each timed replay also times its main kernels
        lib.psf_kernel_timing(1)
        try:
            with torch.cuda.graph(graph):
                run_step()
        finally:
            lib.psf_kernel_timing(0)
        graph.replay()
        torch.cuda.synchronize()
        if psf.device_status() != 0:
            raise RuntimeError("device status after a graph replay is not OK")
    except Exception as exc:  # capture unsupported here: report the eager timing instead
        graph, graph_note = None, f"graph capture failed: {type(exc).__name__}: {exc}"[:200]
    sampler = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    if graph is not None:
        # one replay per step, each bracketed by its own events; after each
        # replay the graph's kernel events are read (the host waits between
        # replays, outside the bracketed region)
        per_step, kacc, kerr = [], {"fwd": [0.0, 0], "bwd": [0.0, 0]}, None
        for _ in range(args.steps):
            per_step += timed(graph.replay, 1)
            if kerr is None:
                try:
                    for name, (tot, n) in kernel_times().items():
                        kacc[name][0] += tot
                        kacc[name][1] += n
                except Exception as exc:  # event nodes not readable: keep the eager kernel times
                    kerr = f"{type(exc).__name__}: {exc}"[:160]
        if kerr is None and kacc["fwd"][1] > 0:
            kt = {name: tuple(v) for name, v in kacc.items()}
            kt_src = "graph replays of the timed region"
        else:
            kt, kt_src = kt_eager, f"eager steps (graph kernel events unavailable: {kerr})"
    else:
        per_step = timed(run_step, args.steps)
        kt, kt_src = kt_eager, "eager steps"
    t1 = time.time()
    if dist:
        dist.barrier()
    clocks = sampler.summary(t0, t1) if sampler else None
    ms = statistics.mean(per_step)
    if psf.device_status() != 0:
        raise RuntimeError("device status after the timed steps is not OK")
    ms_max = max_over_ranks(ms, dist, dev)

    # ---- end to end through the public API: every step copies its inputs in
    # from pinned host memory and its results (out, lse, dq, dk, dv) back out.
    # The steps are pipelined the way a data loader feeds a GPU: step i+1's
    # inputs upload on one copy stream and step i-1's results download on
    # another while step i computes (device inputs double-buffered). No L2
    # flush here: each step's inputs arrive fresh from the host.
    hq, hk, hv, hd = (t.pin_memory() for t in (w.q, w.k, w.v, w.dout))
    host_in = (hq, hk, hv, hd)
    if not dense:
        host_in += (torch.from_numpy(np.ascontiguousarray(w.doc_ids)).pin_memory(),)
    comp_s = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    nbuf = 2
    dev_in = [tuple(torch.empty_like(t) for t in (q, k, v, do) + (() if dense else (ids,))) for _ in range(nbuf)]
    in_ready = [torch.cuda.Event() for _ in range(nbuf)]
    in_free = [torch.cuda.Event() for _ in range(nbuf)]
    out_ready = [torch.cuda.Event() for _ in range(nbuf)]
    out_used = [False] * nbuf
    host_out = [None] * nbuf
    keep = [None] * nbuf
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = 0

    def e2e_step(i):
        nonlocal d2h
        b = i % nbuf
        # The host queues step i only once step i - nbuf's compute is done:
        # this bounds how far the host runs ahead (and so how many steps'
        # results are alive at once) without tying the copies of one step to
        # those of another.
        if out_used[b]:
            in_free[b].synchronize()
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(in_free[b])
            for dst, src in zip(dev_in[b], host_in):
                dst.copy_(src, non_blocking=True)
            in_ready[b].record(h2d_s)
        comp_s.wait_event(in_ready[b])
        dq_, dk_, dv_, dd_ = dev_in[b][:4]
        di_ = None if dense else dev_in[b][4]
        qi_ = None if dense else di_[:, w.q_global_start:w.q_global_start + Lq]
        results = step(dq_, dk_, dv_, dd_, di_, qi_)
        in_free[b].record(comp_s)
        out_ready[b].record(comp_s)
        if host_out[b] is None:
            host_out[b] = [torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in results]
            d2h = sum(r.numel() * r.element_size() for r in results)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(out_ready[b])
            for hdst, r in zip(host_out[b], results):
                r.record_stream(d2h_s)
                hdst.copy_(r, non_blocking=True)
        out_used[b] = True
        keep[b] = results

    for i in range(2 * nbuf):  # warm the pipeline (pinned buffers, the allocator's blocks for in-flight results)
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 50))
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(comp_s)
    h2d_s.wait_event(e_start)
    for i in range(e2e_steps):
        e2e_step(i)
    d2h_done = torch.cuda.Event()
    d2h_done.record(d2h_s)
    comp_s.wait_event(d2h_done)
    e_stop.record(comp_s)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_stop) / e2e_steps, dist, dev)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peak, burst, peak_kind = roofline_peak(*measured_peaks(), ms_max, args.steps)
    # per step: the main kernels' summed launch times (a step may launch a
    # main kernel more than once; its flops are those of all its launches)
    fwd_ms = kt["fwd"][0] / args.steps
    bwd_ms = kt["bwd"][0] / args.steps
    roof = {}
    fwd_name, bwd_name = main_kernels(w.q.shape[-1], w.v.shape[-1])
    for name, kms, kfl, (_, nl) in ((fwd_name, fwd_ms, f_fwd, kt["fwd"]), (bwd_name, bwd_ms, f_bwd, kt["bwd"])):
        ach = kfl / (kms * 1e-3) / 1e12 if kms > 0 else 0.0
        roof[name] = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                      "frac": ach / peak, "frac_of_burst": ach / burst, "ms_per_step": kms,
                      "launches_per_step": nl / args.steps, "algorithmic_tflop_per_step": kfl / 1e12,
                      "timed_in": kt_src,
                      "peak_source": peak_kind}
    dominant = bwd_name if bwd_ms >= fwd_ms else fwd_name
    roofline = dict(roof[dominant])
    roofline["kernel"] = dominant
    roofline["traffic"] = ncu_traffic(dominant, w.name)
    other = [n for n in roof if n != dominant][0]
    roof[other]["traffic"] = ncu_traffic(other, w.name)

    value = whole_job_value(world, flops, ms_max)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.dtype, "data": "synthetic", "impl": "ours",
        "config": config_dict(w, args, pairs, 0 if dense else len(w.extra["lengths"]), world),
        "fwd_tflops": f_fwd / (fwd_ms * 1e-3) / 1e12 if fwd_ms > 0 else None,
        "bwd_tflops": f_bwd / (bwd_ms * 1e-3) / 1e12 if bwd_ms > 0 else None,
        "step_ms_spread": {"min": min(per_step), "median": statistics.median(per_step), "max": max(per_step)},
        "timing": ("each step replayed as one captured CUDA graph" if graph is not None else graph_note),
        "ms_per_step_eager": statistics.mean(eager_steps),
        "kernel_times_from": kt_src,
        "roofline": roofline, "roofline_other": dict(roof[other], kernel=other),
        "e2e": {"value": whole_job_value(world, flops, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
                "timing": "steps pipelined: uploads and downloads overlap neighbouring steps' compute; the host "
                          "queues step i once step i-2's compute is done"},
        "gpu_launches": launches_per_step(dense, bool(split)) * args.steps,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w, args.softcap)
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


def launches_per_step(dense: bool, cross: bool) -> int:
    """Library kernels one step launches: a forward is a preparation kernel and
    the attention kernel, a backward a preparation kernel, the attention kernel
    and the convert kernel; the document path adds the builder; the cross-chunk
    run adds a second document path (local chunk), the cross-chunk builder, a
    second forward and backward, the live-row merge and the live-row dQ add."""
    if dense:
        return 5
    return 6 + (6 + 8 if cross else 0)


def ctypes_double():
    import ctypes

    return ctypes.c_double(0.0)


def ctypes_int():
    import ctypes

    return ctypes.c_int(0)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5,
                    help="workload number: 5 = the headline workload (65536 tokens, D 128, window 4096, plus the "
                         "cross-chunk run); 2 = 8192 tokens, D 128; 3 = dense causal D 512; 4 = 192/128 shard; "
                         "6 = short documents")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--dtype", choices=["bf16", "fp16"], default="bf16",
                    help="16-bit type of q, k, v, dO and the outputs (the headline is bf16)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--softcap", type=float, default=None,
                    help="cap the logits as softcap * tanh(logit / softcap) (off by default)")
    ap.add_argument("--pack-gqa", action=argparse.BooleanOptionalAction, default=True,
                    help="forward and backward with a KV head's query heads packed into one tile where the shape "
                         "allows it (the default; same results, faster on packed documents)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args)
    return our_arm(args)


if __name__ == "__main__":
    sys.exit(main())
