#!/usr/bin/env python3
"""Throughput of batched speculative-decoding verification on GB300.

Metric: verified logit rows/s (B*(K+1) target rows per step for a chain,
B*N for a tree) and the achieved HBM bandwidth on the algorithmic bytes
(every input logit row read once, plus the small index/uniform arrays and
the outputs).

A step is one verification call (all of its kernels) over one batch of
seeded synthetic inputs. Inputs are resident in HBM before timing. Steps cycle
through a pool of input sets whose total size exceeds 4x the L2 cache, so no
step reads inputs another step left in L2. Steps are replayed from CUDA graphs
and timed with CUDA events on the launching stream, bracketed by a barrier and
a device synchronize. One timed repetition is exactly K steps; a workload is
timed as at least five repetitions (more until the repetitions span enough
wall time for the clock sampler) and the median repetition is reported.

The headline line is the long-chain workload (the largest single-GPU
configuration). The same line carries `per_config`: every other workload
timed the same way (at least 200 steps per repetition).

  python bench.py                      # long chain headline + per_config, 1 GPU
  python bench.py --config qwen_sample --steps 2000 --warmup 20 --no-per-config
  python bench.py --impl reference     # the float64 CPU oracle on all host cores
  torchrun --nproc-per-node N bench.py --gpus N   # N independent replicas (weak scaling)

One JSON line is printed by rank 0.
"""

from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

CONFIGS = {
    "llama_greedy": dict(kind="greedy", B=32, K=5, V=128256, dtype="bf16", p_match=0.8, seed=7201,
                         workload="greedy chain verify: Llama-3 vocab V=128256, bf16 logits N(0,3^2), "
                                  "K=5 drafts (6 rows/request), B=32, drafts = row argmax w.p. 0.8"),
    "llama_greedy_b8": dict(kind="greedy", B=8, K=5, V=128256, dtype="bf16", p_match=0.8, seed=7201,
                            workload="greedy chain verify: V=128256 bf16, K=5, B=8"),
    "llama_greedy_b1": dict(kind="greedy", B=1, K=5, V=128256, dtype="bf16", p_match=0.8, seed=7201,
                            workload="greedy chain verify: V=128256 bf16, K=5, B=1"),
    "qwen_sample": dict(kind="sample", B=64, K=4, V=151936, dtype="fp32", seed=7202,
                        workload="stochastic chain verify (exact rule): Qwen vocab V=151936, fp32 target "
                                 "logits N(0,3^2), draft logits = target + N(0,1), T=1, B=64, K=4"),
    "eagle_tree_greedy": dict(kind="tree", B=32, N=64, V=128256, dtype="bf16", T=0.0, rule=0, seed=7203,
                              workload="EAGLE-3 tree verify (greedy): depth 5 / topk 4 pruned to 64 nodes, "
                                       "V=128256 bf16, B=32"),
    "eagle_tree_power": dict(kind="tree", B=32, N=64, V=128256, dtype="bf16", T=1.0, rule=2, alpha=0.3,
                             seed=7203, workload="EAGLE-3 tree verify (power rule alpha=0.3, T=1), "
                                                 "64 nodes, V=128256 bf16, B=32"),
    "eagle_tree_relaxed": dict(kind="tree", B=32, N=64, V=128256, dtype="bf16", T=1.0, rule=1, tau=0.1,
                               seed=7203, workload="EAGLE-3 tree verify (relaxed rule tau=0.1, T=1), "
                                                   "64 nodes, V=128256 bf16, B=32"),
    "long_chain": dict(kind="greedy", B=8, K=4095, V=50257, dtype="bf16", p_match=0.95, seed=7204,
                       workload="long-chain greedy verify: GPT-2 vocab V=50257 bf16, B=8, K+1=4096 rows "
                                "per request, drafts = argmax w.p. 0.95"),
    "llama_greedy_finish": dict(kind="greedy", B=32, K=5, V=128256, dtype="bf16", p_match=0.8, seed=7201,
                                finish=True,
                                workload="greedy chain verify with the finish step: V=128256 bf16, K=5, B=32, "
                                         "a 2-id stop set, per-request max_new in [1, 6], running counters"),
    "long_chain_early": dict(kind="greedy", B=8, K=4095, V=50257, dtype="bf16", p_match=0.95, seed=7204,
                             early=True,
                             workload="long-chain greedy verify with early exit: V=50257 bf16, B=8, K+1=4096 "
                                      "rows per request, drafts = argmax w.p. 0.95; rows after a request's "
                                      "first mismatch are not read"),
    "eagle_tree_build": dict(kind="tree_build", B=32, V=128256, depth=5, topk=4, N=64, dtype="bf16", seed=7205,
                             workload="EAGLE-3 draft-tree construction: depth 5, topk 4, 64 nodes, V=128256 bf16 "
                                      "draft logits N(0,3^2), 17 rank-ordered draft rows per request, B=32"),
    "kv_compact": dict(kind="kv_compact", B=32, N=64, page_size=16, row_elems=65536, dtype="bf16", seed=7206,
                       workload="accepted-path KV compaction: B=32 requests, 64-node trees, paths of 0..5 accepted "
                                "nodes, paged bf16 cache (16 rows per page, 128 KB rows = 32 layers x K,V x 8 "
                                "heads x 128 dims), committed prefixes of 0..256 tokens"),
}
# The verification workloads the HBM-fraction target applies to, then the
# steps before and after verification.
CONTRACT_CONFIGS = ("long_chain", "llama_greedy", "llama_greedy_b8", "llama_greedy_b1", "qwen_sample",
                    "eagle_tree_greedy", "eagle_tree_power", "eagle_tree_relaxed")
NEXT_CONFIGS = ("llama_greedy_finish", "long_chain_early", "eagle_tree_build", "kv_compact")
DEFAULT_CONFIG = "long_chain"
# row pass + decide, plus the draw's two kernels (chunk sums, pick) when a
# call samples; a stochastic chain of at most 16 rows with draft logits and
# the exact rule decides inside the chunk-sum kernel (no decide kernel); a
# stochastic tree call whose rows start on 16-byte boundaries and hold at
# most 48 chunks of 16 KB merges, walks and draws in one cluster kernel
KERNELS_PER_CALL = {"greedy": 2, "sample": 4, "tree": 2, "tree_build": 2, "kv_compact": 1}
FUSED_MAX_ROWS = 16
TREE_CLUSTER_MAX_CHUNKS = 48
FALLBACK_HBM_GBS = 6800.0
MIN_REPS = 5                 # timed repetitions per workload (median reported)
MAX_REPS = 2000
MIN_WINDOW_S = 0.6           # repetitions continue until they span this much wall time
PER_CONFIG_MIN_STEPS = 200   # steps per repetition in per_config
CLOCK_PERIOD_MS = 100


# ------------------------------------------------------------ host helpers

def rank_seed(base, rank):
    """Each rank verifies its own requests (weak scaling): a distinct seed."""
    return int(base) + 1000003 * int(rank)


def reduce_over_ranks(value, op, device, world):
    """MAX or MIN of a per-rank float over all ranks (identity on one rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.MIN)
    return float(t.item())


def aggregate(elapsed_ms_max, rows_per_step, steps, world):
    """Whole-job rows/s from the slowest rank's timed region."""
    return world * rows_per_step * steps / (elapsed_ms_max / 1e3)


# Sources of the kernels one call of each workload kind launches; the entry
# point file (launch shapes) is in every set.
_CALL_SOURCES = {
    "greedy": ("sv_common.cuh", "row_stats.cuh", "decide.cuh", "finish.cuh", "spec_verify.cu"),
    "draw": ("sv_common.cuh", "row_stats.cuh", "decide.cuh", "finish.cuh", "draw.cuh", "rules.cuh",
             "spec_verify.cu"),
    "tree_draw": ("sv_common.cuh", "row_stats.cuh", "decide.cuh", "finish.cuh", "draw.cuh", "rules.cuh",
                  "tree_draw.cuh", "spec_verify.cu"),
    "early": ("sv_common.cuh", "row_stats.cuh", "row_stats_early.cuh", "decide.cuh", "finish.cuh",
              "spec_verify.cu"),
    "tree_build": ("sv_common.cuh", "row_stats.cuh", "tree_build.cuh", "spec_verify.cu"),
    "kv_compact": ("sv_common.cuh", "kv_compact.cuh", "spec_verify.cu"),
}


def source_hash(cfg=None):
    """Hash of the kernel sources behind one call of workload `cfg` (all of
    them when cfg is None). A recorded DRAM capture stays valid only while
    this hash is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_72_gb300", "csrc")
    if cfg is None:
        names = [n for n in sorted(os.listdir(csrc)) if n.endswith((".cu", ".cuh"))]
    else:
        kind = ("early" if cfg.get("early") else cfg["kind"] if cfg["kind"] in ("tree_build", "kv_compact")
                else "draw" if cfg["kind"] == "sample" else "tree_draw" if cfg["kind"] == "tree" and cfg.get("T")
                else "greedy")
        names = sorted(_CALL_SOURCES[kind])
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(config_name):
    """DRAM bytes per call from the committed ncu capture, if it was taken on
    the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic_by_workload.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(config_name)
        if e and e.get("source_hash") == source_hash(CONFIGS[config_name]):
            return float(e["dram_bytes_per_call"])
    except Exception:
        pass
    return None


def metric_name(cfg):
    if cfg["kind"] == "tree_build":
        return "draft logit rows/s (tree construction)"
    if cfg["kind"] == "kv_compact":
        return "KV rows moved/s (accepted-path compaction)"
    return "verified logit rows/s"


def kv_paths(cfg, seed):
    """Synthetic accepted paths: n in 0..5, node ids strictly increasing in 1..N-1."""
    rng = np.random.default_rng(seed)
    B, N = cfg["B"], cfg["N"]
    nodes = np.full((B, 6), -1, dtype=np.int64)
    n = rng.integers(0, 6, size=B)
    for b in range(B):
        nodes[b, 0] = 0
        nodes[b, 1:n[b] + 1] = np.sort(rng.choice(np.arange(1, N), size=n[b], replace=False))
    base = rng.integers(0, 257, size=B)
    return nodes, n, base


def kv_moved_rows(nodes, n):
    return int(sum(1 for b in range(len(n)) for j in range(1, int(n[b]) + 1) if nodes[b, j] != j))


def rows_per_request(cfg):
    """Rows the metric counts for one request of workload `cfg`."""
    if cfg["kind"] == "tree":
        return cfg["N"]
    if cfg["kind"] == "tree_build":
        return 1 + (cfg["depth"] - 1) * cfg["topk"]
    if cfg["kind"] == "kv_compact":
        return None   # data-dependent (the path rows moved)
    return cfg["K"] + 1


def algorithmic_bytes(cfg):
    es = 2 if cfg["dtype"] == "bf16" else 4
    if cfg["kind"] == "kv_compact":   # rows = path rows moved; each read once and written once
        nodes, n, _ = kv_paths(cfg, cfg["seed"])
        rows = kv_moved_rows(nodes, n)
        return rows, 2 * rows * cfg["row_elems"] * es
    B, V = cfg["B"], cfg["V"]
    if cfg["kind"] == "tree_build":   # rows = draft rows; outputs tokens, parents, scores, status
        rows = B * (1 + (cfg["depth"] - 1) * cfg["topk"])
        return rows, rows * V * es + B * cfg["N"] * 12 + B * 4
    if cfg["kind"] == "tree":
        N = cfg["N"]
        W = 6
        rows = B * N
        logits = rows * V * es
        small = B * N * 4 * 2 + (B * N * 4 if cfg.get("T", 0) else 0)
        outs = B * W * (4 + 4 + 4 + 4) + B * 8
        return rows, logits + small + outs
    K = cfg["K"]
    rows = B * (K + 1)
    logits = rows * V * es
    if cfg["kind"] == "sample":
        logits += B * K * V * es
    small = B * K * 4 + (B * (K + 1) * 4 if cfg["kind"] == "sample" else 0)
    outs = B * (K + 1) * 12 + B * 8
    return rows, logits + small + outs


def tree_cluster_path(cfg):
    """Stochastic tree call on the one-kernel cluster path (the bench's rows
    are contiguous and 16-byte aligned, so only the chunk count decides)."""
    if cfg["kind"] != "tree" or not cfg.get("T"):
        return False
    row_bytes = cfg["V"] * (2 if cfg["dtype"] == "bf16" else 4)
    return row_bytes % 16 == 0 and -(-row_bytes // 16384) <= TREE_CLUSTER_MAX_CHUNKS


def launches_per_call(cfg):
    if cfg["kind"] == "sample" and cfg["K"] + 1 <= FUSED_MAX_ROWS:
        return 3
    if tree_cluster_path(cfg):
        return 2
    return KERNELS_PER_CALL[cfg["kind"]] + (2 if cfg["kind"] == "tree" and cfg.get("T") else 0)


def config_dict(cfg, name, world):
    """The `config` object of a result line; the GPU arm and the reference
    arm print the same one for the same workload."""
    rows, alg = algorithmic_bytes(cfg)
    return {"workload": cfg["workload"], "name": name, "B": cfg["B"], "rows_per_step": rows,
            "algorithmic_bytes_per_step": alg,
            "l2_policy": "inputs larger than L2: a rotating pool of input sets totalling more than 4x the L2 "
                         "cache, so no step reads inputs left in L2 by another",
            "timing": f"median of >= {MIN_REPS} repetitions of exactly `steps` steps, each bracketed by a barrier "
                      f"and a device synchronize",
            "parallelism": f"{world} independent replica(s)"}


# ------------------------------------------------------------ clock sampler

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every CLOCK_PERIOD_MS while
    the run lasts; summary(t0, t1) reports the samples inside a wall window."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        # raw samples (SV_CLOCKS_DIR, else the system temp directory); the
        # summaries go into the JSON line
        out_dir = os.environ.get("SV_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_rank_gpu{gpu_index}.csv")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(CLOCK_PERIOD_MS), "-i", str(gpu_index)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def _rows(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                    except ValueError:
                        continue
        except OSError:
            return []
        return rows

    def summary(self, t0, t1):
        if self.proc is None:
            return None
        rows = self._rows()
        if not rows:
            return None
        inside = [r for r in rows if t0 <= r[0] <= t1]
        # no sample inside a short window: the two nearest ones, flagged by samples_in_timed_region = 0
        used = inside if inside else sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:2]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in used])),
                "sm_max_mhz": float(max(r[2] for r in used)),
                "reasons": reasons, "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------ workloads

def make_inputs(cfg, seed, device):
    import torch
    from speculative_decoding_verification_72_gb300 import workloads as W
    dt = torch.bfloat16 if cfg["dtype"] == "bf16" else torch.float32
    if cfg["kind"] == "kv_compact":
        class _Kv:
            pass
        x = _Kv()
        nodes, n, base = kv_paths(cfg, cfg["seed"])   # the same paths in every set: rows/s counts them
        P, B = cfg["page_size"], cfg["B"]
        per_req = (257 + cfg["N"] + P - 1) // P
        g = torch.Generator(device="cpu").manual_seed(seed)
        x.kv = torch.randn((B * per_req, P, cfg["row_elems"]), device=device, dtype=dt)
        x.table = torch.randperm(B * per_req, generator=g).view(B, per_req).to(device=device, dtype=torch.int32)
        x.base = torch.tensor(base, dtype=torch.int32, device=device)
        x.nodes = torch.tensor(nodes, dtype=torch.int32, device=device)
        x.n = torch.tensor(n, dtype=torch.int32, device=device)
        return x
    if cfg["kind"] == "tree_build":
        class _Rows:
            pass
        x = _Rows()
        x.draft_rows = W.draft_tree_rows(B=cfg["B"], V=cfg["V"], depth=cfg["depth"], topk=cfg["topk"], dtype=dt,
                                         seed=seed, device=device)
        return x
    if cfg["kind"] == "greedy":
        x = W.greedy_chain(B=cfg["B"], K=cfg["K"], V=cfg["V"], dtype=dt, p_match=cfg["p_match"],
                           seed=seed, device=device)
        if cfg.get("finish"):   # device-resident finish inputs, so a captured call copies nothing
            g = torch.Generator(device="cpu").manual_seed(seed)
            x.stop_ids = torch.randint(0, cfg["V"], (2,), generator=g).to(device=device, dtype=torch.int32)
            x.max_new = torch.randint(1, cfg["K"] + 2, (cfg["B"],), generator=g).to(device=device,
                                                                                 dtype=torch.int32)
            x.counters = torch.zeros((cfg["B"], 4), dtype=torch.int64, device=device)
        return x
    if cfg["kind"] == "sample":
        return W.stochastic_chain(B=cfg["B"], K=cfg["K"], V=cfg["V"], dtype=dt, seed=seed, device=device)
    return W.eagle_tree(B=cfg["B"], V=cfg["V"], n_nodes=cfg["N"], dtype=dt, seed=seed, device=device)


def call(cfg, x, out=None, ws=None):
    import speculative_decoding_verification_72_gb300 as sv
    if cfg["kind"] == "greedy":
        if cfg.get("early"):
            return sv.spec_verify_greedy_early(x.target, x.draft_tokens, workspace=ws, out=out)
        if cfg.get("finish"):
            return sv.spec_verify_greedy(x.target, x.draft_tokens, workspace=ws, out=out, stop_ids=x.stop_ids,
                                         max_new=x.max_new, counters=x.counters)
        return sv.spec_verify_greedy(x.target, x.draft_tokens, workspace=ws, out=out)
    if cfg["kind"] == "sample":
        return sv.spec_verify_sample(x.target, x.draft_tokens, x.uniforms, draft_logits=x.draft_logits,
                                     workspace=ws, out=out)
    if cfg["kind"] == "tree_build":
        return sv.spec_tree_build(x.draft_rows, cfg["depth"], cfg["topk"], cfg["N"], workspace=ws, out=out)
    if cfg["kind"] == "kv_compact":
        return sv.spec_kv_compact(x.kv, x.table, x.base, x.nodes, x.n, cfg["N"], out=out)
    return sv.spec_verify_tree(x.target, x.node_tokens, x.parents, x.max_depth,
                               temperature=cfg.get("T", 0.0), uniforms=x.uniforms,
                               rule=cfg.get("rule", 0), tau=cfg.get("tau", 0.0),
                               alpha=cfg.get("alpha", 1.0), workspace=ws, out=out)


def input_bytes(x):
    n = 0
    for k in ("target", "draft_logits", "draft_tokens", "uniforms", "node_tokens", "parents", "draft_rows", "kv"):
        t = getattr(x, k, None)
        if t is not None:
            n += t.numel() * t.element_size()
    return n


# ------------------------------------------------------------ CPU oracle
#
# The float64 oracle, as it stands, on a bounded host sample of the workload:
# the same recipe and seed drawn by the CPU generator (`b` whole requests,
# float64 logits). Both CPU legs run before the GPU arm touches CUDA, so the
# all-core leg can fork its workers (which then share the sample
# copy-on-write).

def _mem_available_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def _f64_bytes_per_request(cfg):
    if cfg["kind"] == "kv_compact":
        return ((257 + cfg["N"] + cfg["page_size"] - 1) // cfg["page_size"]) * cfg["page_size"] * cfg["row_elems"] * 8
    rows = rows_per_request(cfg) + (cfg["K"] if cfg["kind"] == "sample" else 0)
    return rows * cfg["V"] * 8


def host_copy(x):
    """float64 / integer NumPy copies of an input set (logits one request at a
    time, so the float32 intermediate stays small)."""
    d = {}
    for k in ("target", "draft_logits", "draft_tokens", "uniforms", "node_tokens", "parents", "draft_rows",
              "kv", "table", "base", "nodes", "n"):
        t = getattr(x, k, None)
        if t is None:
            continue
        if t.is_floating_point():
            a = np.empty(tuple(t.shape), dtype=np.float64)
            for i in range(t.shape[0]):
                a[i] = t[i].float().cpu().numpy()
            d[k] = a
        else:
            d[k] = t.cpu().numpy()
    return d


def cpu_sample(cfg, mem_frac=0.25):
    """(sample config, host arrays): up to B requests, fewer if their float64
    copy would exceed mem_frac of the host's available memory."""
    b = cfg["B"]
    avail = _mem_available_bytes()
    if avail:
        b = max(1, min(b, int(mem_frac * avail // _f64_bytes_per_request(cfg))))
    small = dict(cfg, B=b)
    xh = host_copy(make_inputs(small, cfg["seed"], "cpu"))
    return small, xh


def oracle_request(cfg, xh, r):
    """The oracle on request r of a host sample; returns the rows the metric
    counts for it."""
    from oracle import spec_oracle as O
    sl = slice(r, r + 1)
    if cfg["kind"] == "greedy":
        O.verify_greedy(xh["target"][sl], xh["draft_tokens"][sl])
        return cfg["K"] + 1
    if cfg["kind"] == "sample":
        O.verify_sample(xh["target"][sl], xh["draft_logits"][sl], xh["draft_tokens"][sl], 1.0, xh["uniforms"][sl])
        return cfg["K"] + 1
    if cfg["kind"] == "kv_compact":
        from oracle import kv_compact as KC
        pages = xh["table"][r]                       # this request's pages only
        KC.compact(xh["kv"][pages], np.arange(len(pages))[None], cfg["page_size"], xh["base"][sl],
                   xh["nodes"][sl], xh["n"][sl], cfg["N"])
        return int(xh["n"][r])
    if cfg["kind"] == "tree_build":
        from oracle import tree_build as TB
        TB.build_tree(xh["draft_rows"][sl], cfg["depth"], cfg["topk"], cfg["N"])
        return 1 + (cfg["depth"] - 1) * cfg["topk"]
    O.verify_tree(xh["target"][sl], xh["node_tokens"][sl], xh["parents"][sl], 5, cfg.get("T", 0.0),
                  xh["uniforms"][sl], rule=cfg.get("rule", 0), tau=cfg.get("tau", 0.0), alpha=cfg.get("alpha", 1.0))
    return cfg["N"]


def oracle_one_core(cfg, xh, nreq, budget_s):
    """Requests in turn on this thread until budget_s elapses (at least one).
    Returns (rows/s, requests done)."""
    rows, t_used, done = 0, 0.0, 0
    while t_used < budget_s or done == 0:
        t0 = time.perf_counter()
        rows += oracle_request(cfg, xh, done % nreq)
        t_used += time.perf_counter() - t0
        done += 1
    return rows / t_used, done


def _oracle_worker(cfg, xh, nreq, w, nworkers, conn):
    """Forked worker: on command k, verifies request (w + k * nworkers) mod nreq."""
    os.environ["OMP_NUM_THREADS"] = "1"
    while True:
        k = conn.recv()
        if k is None:
            break
        t0 = time.monotonic()
        rows = oracle_request(cfg, xh, (w + k * nworkers) % nreq)
        conn.send((rows, t0, time.monotonic()))
    conn.close()


class OraclePool:
    """One forked process per host core, each running the oracle on whole
    requests of the host sample. Must be created before any CUDA call."""

    def __init__(self, cfg, xh, nreq, nworkers=None):
        import multiprocessing as mp
        import oracle.spec_oracle  # noqa: F401  (imported before the fork)
        ctx = mp.get_context("fork")
        self.n = nworkers or os.cpu_count() or 1
        self.conns, self.procs = [], []
        for w in range(self.n):
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(cfg, xh, nreq, w, self.n, b), daemon=True)
            p.start()
            b.close()
            self.conns.append(a)
            self.procs.append(p)

    def step(self, k):
        """Every worker verifies one request; returns (rows, wall seconds from
        the first start to the last finish)."""
        for c in self.conns:
            c.send(k)
        res = [c.recv() for c in self.conns]
        return sum(r[0] for r in res), max(r[2] for r in res) - min(r[1] for r in res)

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
                c.close()
            except OSError:
                pass
        for p in self.procs:
            p.join(timeout=10)


def cpu_baseline_prepare(cfg):
    """The host sample and the forked oracle pool, made before any CUDA call;
    the workers wait idle until cpu_baseline_run drives them."""
    small, xh = cpu_sample(cfg)
    nreq = small["B"]
    return {"xh": xh, "nreq": nreq, "pool": OraclePool(cfg, xh, nreq)}


def cpu_baseline_run(cfg, prep, budget_s):
    """The oracle on the prepared host sample: one thread, then every host
    core. Run after the GPU timings: oracle work before them was measured to
    slow the later host-to-device copies of the e2e leg (long chain: 15.9 ms
    per step with no oracle work before, 18.0-18.4 ms after either leg)."""
    xh, nreq, pool = prep["xh"], prep["nreq"], prep["pool"]
    one, done1 = oracle_one_core(cfg, xh, nreq, budget_s)
    rows, wall, k = 0, 0.0, 0
    try:
        while wall < budget_s or k == 0:
            r, t = pool.step(k)
            rows, wall, k = rows + r, wall + t, k + 1
    finally:
        pool.close()
    sample = (f"{nreq} of {cfg['B']} requests of the workload's recipe drawn on the host (seed {cfg['seed']}), "
              f"float64 NumPy oracle")
    return {"value": rows / wall, "unit": "rows/s", "cores": pool.n, "kind": "oracle",
            "sample": f"{sample}; {pool.n} forked processes, one request each per round, {k} rounds "
                      f"(~{wall:.0f} s)",
            "one_core": {"value": one, "unit": "rows/s", "cores": 1,
                         "sample": f"{sample}; one thread, {done1} requests (~{budget_s:.0f} s)"},
            "host_cores": os.cpu_count()}


def run_reference(args, cfg, name):
    """Reference arm: the float64 CPU oracle, as it stands, on every host core.
    A step is one round of the oracle pool (each process verifies one whole
    request of the host sample)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    if rank != 0:
        return 0
    steps = args.steps if args.steps is not None else 20
    warmup = args.warmup if args.warmup is not None else 3
    small, xh = cpu_sample(cfg)
    nreq = small["B"]
    pool = OraclePool(cfg, xh, nreq)
    try:
        for w in range(warmup):
            pool.step(w)
        total_rows, total_t = 0, 0.0
        for s in range(steps):
            r, t = pool.step(warmup + s)
            total_rows, total_t = total_rows + r, total_t + t
    finally:
        pool.close()
    value = total_rows / total_t
    sample = (f"{nreq} of {cfg['B']} requests of the workload's recipe drawn on the host (seed {cfg['seed']}); "
              f"each step: {pool.n} forked processes verify one whole request each, float64 NumPy oracle")
    line = {
        "impl": "reference", "metric": metric_name(cfg), "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warmup,
        "ms_per_step": 1e3 * total_t / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; shapes from the pages, no dataset or weights)",
        "config": config_dict(cfg, name, world),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": pool.n, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ GPU arm

def _workspace_need(cfg):
    import speculative_decoding_verification_72_gb300 as sv
    lib = sv.load_library()
    dt = 1 if cfg["dtype"] == "bf16" else 0
    if cfg["kind"] == "greedy":
        return lib.spec_verify_greedy_workspace_size(cfg["B"], cfg["K"], cfg["V"], dt)
    if cfg["kind"] == "sample":
        return lib.spec_verify_sample_workspace_size(cfg["B"], cfg["K"], cfg["V"], dt, 1)
    if cfg["kind"] == "tree_build":
        return lib.spec_tree_build_workspace_size(cfg["B"], cfg["depth"], cfg["topk"], cfg["V"])
    if cfg["kind"] == "kv_compact":
        return 256
    return lib.spec_verify_tree_workspace_size(cfg["B"], cfg["N"], cfg["V"], dt)


class GpuWorkload:
    """One workload on this rank's GPU: a rotating pool of input sets larger
    than 4x L2, caller-owned outputs and workspace, and CUDA graphs of calls."""

    def __init__(self, cfg, name, dev, rank, stream):
        import torch
        self.cfg, self.name, self.dev, self.stream = cfg, name, dev, stream
        self.rows, self.alg_bytes = algorithmic_bytes(cfg)
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20) or (126 << 20)
        first = make_inputs(cfg, rank_seed(cfg["seed"], rank), dev)
        self.set_bytes = input_bytes(first)
        self.nsets = max(2, min(512, math.ceil(4 * l2 / self.set_bytes)))
        self.pool = [first] + [make_inputs(cfg, rank_seed(cfg["seed"] + 17 * i, rank), dev)
                               for i in range(1, self.nsets)]
        self.out = call(cfg, self.pool[0])
        self.ws = torch.empty(max(1 << 20, _workspace_need(cfg)), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        self.per_graph = self.nsets * max(1, math.ceil(32 / self.nsets))
        self.graphs = {}
        self.pool_desc = (f"{self.nsets} input sets, {self.nsets * self.set_bytes / 1e6:.0f} MB "
                          f"> 4x L2 ({l2 / 1e6:.0f} MB); graphs of up to {self.per_graph} calls")

    def graph_of(self, n):
        import torch
        if n not in self.graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                for i in range(n):               # warm the capture stream
                    call(self.cfg, self.pool[i % self.nsets], out=self.out, ws=self.ws)
                self.stream.synchronize()
                with torch.cuda.graph(g, stream=self.stream):
                    for i in range(n):
                        call(self.cfg, self.pool[i % self.nsets], out=self.out, ws=self.ws)
            torch.cuda.synchronize()
            self.graphs[n] = g
        return self.graphs[n]

    def replay(self, steps):
        """Enqueue exactly `steps` calls on self.stream."""
        full, rem = divmod(steps, self.per_graph)
        for _ in range(full):
            self.graph_of(self.per_graph).replay()
        if rem:
            self.graph_of(rem).replay()

    def prepare(self, steps, warmup):
        import torch
        full, rem = divmod(steps, self.per_graph)
        if full:
            self.graph_of(self.per_graph)
        if rem:
            self.graph_of(rem)
        with torch.cuda.stream(self.stream):
            self.replay(max(3, warmup))
        torch.cuda.synchronize()

    def bytes_read_per_call(self):
        """Early exit: logit bytes the library reports it read, mean over the pool."""
        tot = 0
        for x in self.pool:
            r = call(self.cfg, x, out=self.out, ws=self.ws)
            tot += int(r["bytes_read"].item())
        return tot / len(self.pool)


def time_workload(wl, steps, world, sampler):
    """Repetitions of exactly `steps` calls, each bracketed by a barrier and a
    device synchronize and timed with CUDA events on the launch stream (the
    slowest rank's time per repetition). At least MIN_REPS repetitions, more
    until they span MIN_WINDOW_S of wall time."""
    import torch
    import torch.distributed as dist
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    reps_ms, nreps, t_first, t_last = [], MIN_REPS, None, None
    while len(reps_ms) < nreps:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        tw0 = time.time()
        with torch.cuda.stream(wl.stream):
            e0.record(wl.stream)
            wl.replay(steps)
            e1.record(wl.stream)
        torch.cuda.synchronize()
        tw1 = time.time()
        if world > 1:
            dist.barrier()
        t_first = tw0 if t_first is None else t_first
        t_last = tw1
        reps_ms.append(reduce_over_ranks(e0.elapsed_time(e1), "max", wl.dev, world))
        if len(reps_ms) == 1:
            rep_wall = reduce_over_ranks(tw1 - tw0, "max", wl.dev, world)
            nreps = int(min(MAX_REPS, max(MIN_REPS, math.ceil(MIN_WINDOW_S / max(rep_wall, 1e-6)))))
    med = float(np.median(reps_ms))
    return {"ms_per_step": med / steps, "elapsed_ms": med, "steps": steps, "reps": len(reps_ms),
            "rep_ms": {"min": float(min(reps_ms)), "median": med, "max": float(max(reps_ms))},
            "window_s": t_last - t_first, "clocks": sampler.summary(t_first, t_last) if sampler else None}


def kernel_desc(cfg):
    if cfg.get("early"):
        d = "one verify call: row_stats_early_kernel (bytes it read) + decide kernel"
    elif cfg["kind"] == "tree_build":
        d = "one build call: row_topk_kernel (all draft logit bytes) + tree_select_kernel"
    elif cfg["kind"] == "kv_compact":
        d = "one compaction call: kv_compact_kernel (path rows read + written)"
    elif tree_cluster_path(cfg):
        d = ("one verify call: row_stats_kernel (all logit bytes) + tree_walk_draw_kernel (row merges, walk "
             "and draw, one cluster of 8 CTAs per request)")
    elif launches_per_call(cfg) == 3:
        d = "one verify call: row_stats_kernel (all logit bytes) + draw kernels (chunk sums with the decision, pick)"
    else:
        d = "one verify call: row_stats_kernel (all logit bytes) + decide kernel"
    return d + (" + draw kernels (chunk sums, pick)" if launches_per_call(cfg) == 4 else "")


def roofline(cfg, name, ms_per_step, read_bytes=None):
    """Bandwidth roofline of one call: algorithmic bytes (or the bytes an early
    exit actually read) over the event-timed duration of the whole call, so
    a lower bound on the row-statistics kernel's own rate."""
    peak, kind = measured_peak()
    _, alg = algorithmic_bytes(cfg)
    achieved = (read_bytes if read_bytes is not None else alg) / (ms_per_step / 1e3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if kind == "measured" else "fallback 6.8 TB/s",
            "kernel": kernel_desc(cfg),
            "traffic": recorded_traffic(name) if cfg["B"] == CONFIGS[name]["B"] else None}


def per_config_entry(wl, t, world):
    cfg = wl.cfg
    rb = wl.bytes_read_per_call() if cfg.get("early") else None
    e = {"workload": cfg["workload"], "metric": metric_name(cfg),
         "value": aggregate(t["elapsed_ms"], wl.rows, t["steps"], world), "unit": "rows/s",
         "ms_per_step": t["ms_per_step"], "steps": t["steps"], "reps": t["reps"], "rep_ms": t["rep_ms"],
         "rows_per_step": wl.rows, "algorithmic_bytes_per_step": wl.alg_bytes,
         "roofline": roofline(cfg, wl.name, t["ms_per_step"], rb), "clocks": t["clocks"],
         "gpu_launches_per_step": launches_per_call(cfg), "pool": wl.pool_desc,
         "contract": wl.name in CONTRACT_CONFIGS}
    if rb is not None:
        e["bytes_read_per_step"] = rb
        e["roofline_bytes"] = "bytes actually read (library-reported), not all logit bytes"
    return e


def _e2e_greedy_host(cfg, x, dev, steps):
    """Plain greedy chains: the host-buffer entry point (spec_verify_greedy_host)
    on page-locked inputs and outputs. Each step copies the step's logits in
    groups, verifies each group as it lands, reads the outputs back and
    synchronizes."""
    import torch
    import speculative_decoding_verification_72_gb300 as sv
    lib = sv.load_library()
    xh = x.target.cpu().pin_memory()
    dh = x.draft_tokens.cpu().pin_memory()
    B, R, V = xh.shape
    outh = dict(tokens=torch.empty((B, R), dtype=torch.int32).pin_memory(),
                num_accepted=torch.empty((B,), dtype=torch.int32).pin_memory(),
                logprob=torch.empty((B, R), dtype=torch.float32).pin_memory(),
                mu=torch.empty((B, R), dtype=torch.float32).pin_memory(),
                status=torch.empty((B,), dtype=torch.int32).pin_memory())
    dt = 1 if xh.dtype == torch.bfloat16 else 0
    ws = torch.empty(lib.spec_verify_greedy_host_workspace_size(B, R - 1, V, dt, 0), dtype=torch.uint8, device=dev)
    h2d = xh.numel() * xh.element_size() + dh.numel() * dh.element_size()
    d2h = sum(v.numel() * v.element_size() for v in outh.values())
    n = max(3, min(steps, 300))

    def one():
        sv.spec_verify_greedy_host(xh, dh, workspace=ws, out=outh)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        one()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    rows, _ = algorithmic_bytes(cfg)
    return {"value": rows / (ms / 1e3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n, "ms_per_step": ms,
            "api": "spec_verify_greedy_host (page-locked host logits, copies overlapped with verification)"}


def _e2e(cfg, x, dev, steps, out, ws):
    """Same metric through the public API with host buffers: every step copies
    that step's inputs from pinned host memory and reads the results back."""
    import torch
    if cfg["kind"] == "greedy" and not cfg.get("early") and not cfg.get("finish"):
        return _e2e_greedy_host(cfg, x, dev, steps)
    names = [k for k in ("target", "draft_logits", "draft_tokens", "uniforms", "node_tokens", "parents",
                         "stop_ids", "max_new", "draft_rows", "table", "base", "nodes", "n")
             if getattr(x, k, None) is not None]
    host = {k: getattr(x, k).cpu().pin_memory() for k in names}
    devb = {k: torch.empty_like(getattr(x, k)) for k in names}
    outh = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in outh.values())
    n = max(3, min(steps, 300))

    class Inp:
        pass

    inp = Inp()
    for k in ("target", "draft_logits", "draft_tokens", "uniforms", "node_tokens", "parents",
              "stop_ids", "max_new", "draft_rows", "table", "base", "nodes", "n"):
        setattr(inp, k, devb.get(k))
    inp.kv = getattr(x, "kv", None)               # the KV cache is device-resident state
    inp.max_depth = getattr(x, "max_depth", None)
    inp.counters = getattr(x, "counters", None)   # running totals stay on the device

    def one():
        for k in names:
            devb[k].copy_(host[k], non_blocking=True)
        res = call(cfg, inp, out=out, ws=ws)
        for k in outh:
            outh[k].copy_(res[k], non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        one()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    rows, _ = algorithmic_bytes(cfg)
    return {"value": rows / (ms / 1e3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n, "ms_per_step": ms,
            "api": "device entry point, inputs copied from page-locked host memory each step"}


def run_gpu(args, cfg, name):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    steps = args.steps if args.steps is not None else 200
    warmup = max(3, args.warmup if args.warmup is not None else 20)

    # The CPU oracle legs' sample and forked pool are made first (the fork
    # must happen before this process makes any CUDA call); the legs run after
    # the GPU timings.
    cpu_prep = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_prep = cpu_baseline_prepare(cfg)

    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    import speculative_decoding_verification_72_gb300 as sv
    sv.load_library()
    stream = torch.cuda.Stream(device=dev)
    sampler = ClockSampler(local)
    time.sleep(0.3)

    # headline workload: exactly `steps` calls per repetition
    wl = GpuWorkload(cfg, name, dev, rank, stream)
    wl.prepare(steps, warmup)
    t = time_workload(wl, steps, world, sampler)
    value = aggregate(t["elapsed_ms"], wl.rows, steps, world)
    read_bytes = wl.bytes_read_per_call() if cfg.get("early") else None
    roof = roofline(cfg, name, t["ms_per_step"], read_bytes)
    per_config = {}
    want_per_config = world == 1 and not args.no_per_config
    if want_per_config:
        if steps >= PER_CONFIG_MIN_STEPS:
            per_config[name] = per_config_entry(wl, t, world)
        else:
            wl.prepare(PER_CONFIG_MIN_STEPS, 0)
            per_config[name] = per_config_entry(wl, time_workload(wl, PER_CONFIG_MIN_STEPS, world, sampler), world)
    e2e = _e2e(cfg, wl.pool[0], dev, steps, wl.out, wl.ws)
    if world > 1:   # the slowest replica's rate, times the replicas
        e2e["value"] = reduce_over_ranks(e2e["value"], "min", dev, world) * world
    pool_desc = wl.pool_desc
    del wl
    torch.cuda.empty_cache()

    if want_per_config:
        for other in CONTRACT_CONFIGS + NEXT_CONFIGS:
            if other == name:
                continue
            ow = GpuWorkload(CONFIGS[other], other, dev, rank, stream)
            n_steps = max(steps, PER_CONFIG_MIN_STEPS)
            ow.prepare(n_steps, warmup)
            per_config[other] = per_config_entry(ow, time_workload(ow, n_steps, world, sampler), world)
            del ow
            torch.cuda.empty_cache()
    time.sleep(0.3)
    sampler.stop()
    cpu = cpu_baseline_run(cfg, cpu_prep, args.cpu_budget) if cpu_prep is not None else None

    line = {
        "metric": metric_name(cfg), "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": t["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if cfg["dtype"] == "bf16" else "f32",
        "data": "synthetic (seeded; shapes from the pages, no dataset or weights)",
        "config": config_dict(cfg, name, world),
        "repetitions": {"count": t["reps"], "rep_ms": t["rep_ms"], "reported": "median repetition",
                        "window_s": t["window_s"], "pool": pool_desc},
        "hbm_gbs": roof["achieved"],
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": steps * launches_per_call(cfg) * t["reps"],
        "gpu_launches_per_step": launches_per_call(cfg),
        "clocks": t["clocks"],
        "per_config": per_config or None,
    }
    if read_bytes is not None:
        line["config"]["bytes_read_per_step"] = read_bytes
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(CONFIGS), default=DEFAULT_CONFIG)
    ap.add_argument("--cpu-budget", type=float, default=8.0,
                    help="seconds of oracle work for each cpu_baseline leg (one core, all cores)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="time only the --config workload")
    ap.add_argument("--batch", type=int, default=None,
                    help="requests per call for the --config workload (a smaller case for profiling; "
                         "the workload string records it)")
    args = ap.parse_args(argv)
    cfg = CONFIGS[args.config]
    if args.batch is not None:
        if args.batch < 1:
            ap.error("--batch must be >= 1")
        cfg = dict(cfg, B=args.batch, workload=f"{cfg['workload']} [batch overridden: B={args.batch}]")
    if args.impl == "reference":
        return run_reference(args, cfg, args.config)
    return run_gpu(args, cfg, args.config)


if __name__ == "__main__":
    sys.exit(main())
