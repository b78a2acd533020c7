"""Benchmark of the tree-verification hot path on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one whole pass of the hot path over one batch of synthetic input:
depth + 1 levels of draft top-k expansion, the final total_tokens selection, the
tree metadata, tree-verification attention of one layer (RoPE, KV append, split-KV
attention, merge) and the greedy acceptance with KV compaction. Inputs are resident
in HBM before the timed region; the step is replayed from a CUDA graph; L2 is flushed
(a 256 MiB write) between timed launches. The JSON line reports steps/s (whole job),
the per-call times, the roofline of the attention call against MEASURED_PEAKS.json,
an end-to-end number through host buffers, and the CPU oracle as a baseline. An
attention or top-k leg whose inputs are larger than L2 is also replayed as four calls
back to back in one graph (each call streams its inputs from HBM, so no flush is needed
between them); its roofline takes that per-call time (the time inside a step, without
the launch latency of a graph of one call) and keeps the one-call figure beside it
(us_per_launch_alone, frac_alone).

The default workload is long70b (batch 4, prefix 32768, 70B-shaped heads: the largest
single-GPU shape, a long-prefix one). In the same timed loop the attention call of the
serving mix and of the large-batch sweep (65-node trees) and the sweep's top-k level
([640, 128256] fp32 logits) are replayed, each after its own L2 flush, and reported as
roofline_attn_serving, roofline_attn_sweep and roofline_topk_sweep (--no-side leaves
them out).

--impl reference times the CPU oracle (the reference arm: a deliberately slow,
obviously correct restatement of the method) on the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "tree-verify attn µs/layer, achieved HBM GB/s and % roofline; top-k rows/s"
UNIT = "layer-verify steps/s"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 * 10 ** 6  # GB300 L2
CHAIN = 4  # calls per chained graph of a leg whose inputs exceed L2


def plain(x):
    """JSON-safe copy (numpy scalars -> Python numbers)."""
    if isinstance(x, dict):
        return {k: plain(v) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [plain(v) for v in x]
    if isinstance(x, np.generic):
        return x.item()
    return x


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for about 2 s of timed work, at least 50)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long70b", choices=sorted(W.WORKLOADS))
    ap.add_argument("--total-tokens", type=int, default=0)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="time only the chosen workload (no serving / sweep side legs)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    return ap.parse_args()


def max_over_ranks(values, world: int):
    """The element-wise maximum of `values` over all ranks (every rank gets it): the
    replicas agree on a step count and report the slowest rank's times. A plain list at
    world size 1; a CUDA tensor for NCCL, a CPU one for gloo."""
    if world <= 1:
        return [float(x) for x in values]
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def workload(args):
    w = W.WORKLOADS[args.workload]
    if args.total_tokens:
        w = w.with_(total_tokens=args.total_tokens)
    if w.fixed_parents is not None:
        raise SystemExit("the bench runs dynamic-tree workloads")
    return w


def algorithmic(w, prefix, depths_per_req, esize=2):
    """Algorithmic bytes and FLOPs of one tree_verify_attn call.

    bytes: KV prefix read once per KV head, the tree's new k/v read and written to the
    cache, q read and out written. FLOPs: 4 * D per visible (query head, key) pair.
    """
    hkv, hq, d = w.num_kv_heads, w.num_q_heads, w.head_dim
    nbytes = 0
    flops = 0
    for p, deps in zip(prefix, depths_per_req):
        p, t = int(p), len(deps)  # Python ints: the FLOP count overflows 32 bits
        nbytes += 2 * p * hkv * d * esize + 4 * t * hkv * d * esize + 2 * t * hq * d * esize
        flops += 4 * d * hq * sum(p + dep + 1 for dep in deps)
    return nbytes, flops


PROFILES = os.path.join(ROOT, "profiles")


def source_digest(paths):
    """sha256 over the named source files (repository-relative), in order."""
    import hashlib
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic(kernel, workload):
    """DRAM bytes (read + write) of one launch of `kernel` on `workload` from the ncu
    capture recorded in profiles/traffic.json, with the summary that holds it; (None,
    reason) when there is no capture, or the kernel's sources have changed since."""
    path = os.path.join(PROFILES, "traffic.json")
    if not os.path.exists(path):
        return None, "no capture"
    with open(path) as f:
        entries = json.load(f)["entries"]
    for e in entries:
        if e["kernel"] == kernel and e["workload"] == workload:
            if source_digest(e["sources"]) != e["sources_sha256"]:
                return None, f"kernel changed since the capture in {e['summary']}"
            return int(e["dram_read"] + e["dram_write"]), e["summary"]
    return None, "no capture"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return m["hbm_gbs"], m["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling (every 50 ms, with timestamps) around the timed region; only
    the samples taken inside the region's wall-clock window count."""

    def __init__(self, out):
        self.out = out
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
                 "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "50", "-i",
                 os.environ.get("LOCAL_RANK", "0")],
                stdout=open(self.out, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        # the sampler is running (it has written a sample) before the region starts
        t = time.time()
        while self.proc and time.time() - t < 5.0:
            if os.path.exists(self.out) and os.path.getsize(self.out) > 0:
                break
            time.sleep(0.02)
        return self

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        time.sleep(0.1)  # the sample that covers the region's end

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=10)
            except subprocess.TimeoutExpired:  # a sampler stuck in the driver: leave it
                self.proc.kill()

    def summary(self):
        if not os.path.exists(self.out) or self.t0 is None or self.t1 is None:
            return None
        import datetime
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.out):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, cmax = float(f[2]), float(f[3])
            except ValueError:
                continue
            if not (self.t0 - 0.05 <= ts <= self.t1 + 0.05):
                continue
            sm.append(clk)
            mx.append(cmax)
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------------------
# Side legs: the attention call of other workloads (and the sweep's top-k level), timed
# in the same loop as the main workload so one run reports every long-prefix roofline.
SIDE_LEGS = (("serving", ("attn",)), ("sweep", ("attn", "topk")))


def kv_cache(w, dev, gen, T, cap):
    """Random (already rotated) KV cache of the workload: contiguous [B, Hkv, cap, D] or
    paged [pool, Hkv, 64, D] behind the workload's block table."""
    import torch
    if w.paged:
        table, pool = W.block_table(w, cap)
        shp = (pool, w.num_kv_heads, 64, w.head_dim)
        kc = (torch.randn(*shp, device=dev, generator=gen) * w.scale).to(torch.bfloat16)
        vc = (torch.randn(*shp, device=dev, generator=gen) * w.scale).to(torch.bfloat16)
        return T.KVCache(kc, vc, torch.from_numpy(table).to(dev))
    shp = (w.batch, w.num_kv_heads, cap, w.head_dim)
    kc = (torch.randn(*shp, device=dev, generator=gen) * w.scale).to(torch.bfloat16)
    vc = (torch.randn(*shp, device=dev, generator=gen) * w.scale).to(torch.bfloat16)
    return T.KVCache(kc, vc)


def tree_depths(parents_rows):
    out = []
    for pars in parents_rows:
        d = []
        for p in pars:
            d.append(0 if p < 0 else d[p] + 1)
        out.append(d)
    return out


def side_state(name, legs, dev, gen, T):
    """Inputs in HBM for one side workload: its trees from the expansion of its own
    seeded draft logits, their metadata, q/k/v and a KV cache; returns the legs as
    callables with what their rooflines need."""
    import torch
    w = W.WORKLOADS[name]
    b, k = w.batch, w.top_k
    prefix = W.prefix_lengths(w)
    t_max = w.num_nodes
    cap = int(math.ceil((w.max_prefix + t_max + 16) / 64) * 64)
    cache = kv_cache(w, dev, gen, T, cap)
    shape = T.TreeShape(b, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_prefix,
                        vocab=w.vocab, top_k=k, depth=w.depth, total_tokens=w.total_tokens)
    hp = T.HotPath(shape, cache)
    levels = [torch.from_numpy(W.draft_logits_batch(w, lvl)).to(dev)
              for lvl in range(1, w.depth + 2)]
    root = torch.from_numpy(W.root_tokens(w)).to(dev)
    prefix_t = torch.from_numpy(prefix).to(dev)
    hp.expand(levels, root)
    hp.build_meta(prefix_t)
    torch.cuda.synchronize()
    depths = tree_depths(hp.parents.cpu().numpy())
    q, k_new, v_new = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in W.new_qkv(w))
    sm_scale = 1.0 / math.sqrt(w.head_dim)
    fns = {}
    if "attn" in legs:
        fns["attn_" + name] = lambda: hp.verify(q, k_new, v_new, prefix_t, w.theta, sm_scale)
    if "topk" in legs:
        lvl_out = hp.front[1]
        fns["topk_" + name] = lambda: T.draft_topk_expand(
            levels[1], k, 2, hp.front[0][1], hp.front[0][2], hp.store_token, hp.store_score,
            hp.store_parent, *lvl_out, hp.topk_ws)
    # keep the inputs alive with the callables
    return {"w": w, "prefix": prefix, "depths": depths, "fns": fns, "hp": hp,
            "keep": (levels, root, q, k_new, v_new, prefix_t, cache),
            "attn_launches": hp.attn_kernels()}


def attn_roofline(w, prefix, depths, us, hbm, tf, src):
    """Roofline of one tree_verify_attn call (SURVEY-style algorithmic bytes / FLOPs)."""
    nbytes, flops = algorithmic(w, prefix, depths)
    s = us / 1e6
    t_hbm, t_tc = nbytes / (hbm * 1e9), flops / (tf * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    if bound == "hbm":
        achieved, peak, unit = nbytes / s / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit = flops / s / 1e12, tf, "TFLOP/s"
    tr, tr_src = traffic("attn", w.name)
    return {"kernel": f"tree_verify_attn on {w.name} (prep + tcgen05 split-KV attention + "
                      "split merge)",
            "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_source": src, "traffic": tr, "traffic_source": tr_src,
            "algorithmic_bytes": nbytes, "algorithmic_flops": flops, "us_per_launch": us,
            "roofline_us": max(t_hbm, t_tc) * 1e6, "hbm_GBps": nbytes / s / 1e9,
            "nodes_kv_tokens_per_s": sum(len(d) * (int(p) + len(d))
                                         for p, d in zip(prefix, depths)) / s}


def topk_roofline(w, us, hbm, src):
    """Roofline of one expansion level: every frontier row's fp32 logits read once."""
    rows = w.batch * w.top_k
    nbytes = rows * w.vocab * 4
    gbps = nbytes / (us / 1e6) / 1e9
    tr, tr_src = traffic("topk", w.name)
    return {"kernel": f"draft_topk_expand level on {w.name} ({rows} rows x {w.vocab} fp32)",
            "bound": "hbm", "achieved": gbps, "peak": hbm, "unit": "GB/s", "frac": gbps / hbm,
            "peak_source": src, "traffic": tr, "traffic_source": tr_src,
            "algorithmic_bytes": nbytes, "us_per_launch": us,
            "rows_per_s": rows / (us / 1e6)}


# --------------------------------------------------------------------------------------
def native(args):
    import torch
    import torch.distributed as dist

    import tree_speculative_decoding_verify_gb300 as T
    from tree_speculative_decoding_verify_gb300 import build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload(args)
    b, k, v = w.batch, w.top_k, w.vocab
    prefix = W.prefix_lengths(w)
    p_max = w.max_prefix
    paged = w.paged
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + rank)

    # ---- inputs resident in HBM ------------------------------------------------------
    levels = [torch.from_numpy(W.draft_logits_batch(w, lvl)).to(dev) for lvl in range(1, w.depth + 2)]
    root = torch.from_numpy(W.root_tokens(w)).to(dev)
    q, k_new, v_new = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in W.new_qkv(w))
    t_max = w.num_nodes
    # room for the verified tree and for the drafter leg's grown tree (1 + K (depth + 1)
    # nodes), each rounded up to 16 slots past the prefix
    cap = int(math.ceil((p_max + max(t_max, 1 + k * (w.depth + 1)) + 16) / 64) * 64)
    scale = w.scale
    cache = kv_cache(w, dev, gen, T, cap)
    shape = T.TreeShape(b, w.num_q_heads, w.num_kv_heads, w.head_dim, p_max, vocab=v, top_k=k,
                        depth=w.depth, total_tokens=w.total_tokens)
    hp = T.HotPath(shape, cache)
    prefix_t = torch.from_numpy(prefix).to(dev)
    sm_scale = 1.0 / math.sqrt(w.head_dim)

    # the tree the expansion builds (deterministic) -> planted target argmax
    hp.expand(levels, root)
    torch.cuda.synchronize()
    toks = hp.tokens.cpu().numpy()
    pars = hp.parents.cpu().numpy()
    target = np.stack([W.plant_target(w, i, toks[i], pars[i]) for i in range(b)])
    target_t = torch.from_numpy(target).to(dev)
    depths = tree_depths(pars)

    def step():
        hp.step(levels, root, q, k_new, v_new, prefix_t, target_t, w.theta, sm_scale)

    def attn():
        hp.verify(q, k_new, v_new, prefix_t, w.theta, sm_scale)

    lvl_ws = hp.topk_ws
    lvl_out = hp.front[1]

    # the target's lm_head over every node of the batch (the greedy token per node)
    lm_h, lm_v = W.TARGET_LM_HEAD[w.name]
    lm_rows = b * t_max
    lm_hidden = torch.from_numpy(W.lm_head_hidden(w, lm_rows, lm_h)).to(torch.bfloat16).to(dev)
    lm_weight = torch.empty(lm_v, lm_h, dtype=torch.bfloat16, device=dev)
    for v0, blk in W.lm_head_weight_blocks(w, lm_v, lm_h):
        lm_weight[v0:v0 + blk.shape[0]] = torch.from_numpy(blk).to(torch.bfloat16).to(dev)
    lm_argmax = torch.zeros(lm_rows, dtype=torch.int32, device=dev)
    lm_ws = torch.empty(max(T.lm_head_argmax_workspace_size(lm_rows, lm_v), 256),
                        dtype=torch.uint8, device=dev)

    def lm_head():
        T.lm_head_argmax(lm_hidden, lm_weight, lm_argmax, lm_ws)

    # non-greedy acceptance over the same trees: nucleus sampling (temperature 0.8,
    # top-p 0.9) on the target's logits at every node, the rejection walk, compaction
    hp.build_meta(prefix_t)
    torch.cuda.synchronize()
    sa_v = lm_v
    nodes = hp.num_nodes.cpu().numpy()
    sa_logits = torch.from_numpy(np.stack([
        W.target_logits(w, i, toks[i][:nodes[i]], pars[i][:nodes[i]], sa_v, t_max)
        for i in range(b)])).to(dev)
    uni = np.stack([W.uniforms(w, i, t_max) for i in range(b)])
    sa_u = torch.from_numpy(np.ascontiguousarray(uni[:, :t_max])).to(dev)
    sa_uf = torch.from_numpy(np.ascontiguousarray(uni[:, t_max])).to(dev)
    sa_prm = (torch.full((b,), 0.8, device=dev), torch.zeros(b, dtype=torch.int32, device=dev),
              torch.full((b,), 0.9, device=dev), torch.zeros(b, device=dev))
    sa_out = [torch.zeros(b, shape.max_depth + 1, dtype=torch.int32, device=dev),
              torch.zeros(b, dtype=torch.int32, device=dev),
              torch.zeros(b, dtype=torch.int32, device=dev),
              torch.zeros(b, shape.max_depth + 1, 2, dtype=torch.int32, device=dev),
              torch.zeros(b, dtype=torch.int32, device=dev)]
    sa_ws = torch.empty(T.tree_sample_accept_workspace_size(b, t_max), dtype=torch.uint8,
                        device=dev)

    # expansion variants: one level with probability-product scores, the d2t id map over
    # the tree, one fixed-branching level (every frontier row of the level's logits,
    # width 2)
    d2t = torch.from_numpy(np.random.default_rng(5).permutation(lm_v)[:v].astype(np.int32)).to(dev)
    fx_tok = torch.zeros(b, 1 + k * 2 + k, dtype=torch.int32, device=dev)
    fx_par = torch.zeros_like(fx_tok)
    map_tok = hp.tokens.clone()

    def topk_product():
        T.draft_topk_expand(levels[1], k, 2, hp.front[0][1], hp.front[0][2], hp.store_token,
                            hp.store_score, hp.store_parent, *lvl_out, lvl_ws, product=True)

    def variants():
        map_tok.copy_(hp.tokens)
        T.draft_to_target(map_tok, hp.num_nodes, d2t)
        T.draft_fixed_level(levels[1], 2, 1 + k, 1, fx_tok, fx_par)

    # drafter-side tree attention: the drafter's mask grown to its last level (1 + K
    # (depth + 1) nodes, each level's parents in the level before), then the tree
    # attention of all its nodes over it (the drafter's layer has the target's head shape)
    dn = 1 + k * (w.depth + 1)
    dmask = torch.zeros(b, dn, (dn + 31) // 32, dtype=torch.int32, device=dev)
    dpos = torch.zeros(b, dn, dtype=torch.int32, device=dev)
    dparents = [-1]
    n0, last = 1, None
    for lvl in range(w.depth + 1):
        front = [0] if lvl == 0 else list(range(n0 - k, n0))
        par = [front[j % len(front)] for j in range(k)]
        dparents += par
        last = (n0, torch.tensor([par] * b, dtype=torch.int32, device=dev))
        T.draft_grow_mask(dmask, dpos, last[1], prefix_t, n0)
        n0 += k
    d_depth = [0]
    for pp in dparents[1:]:
        d_depth.append(d_depth[pp] + 1)
    dq = (torch.randn(b, dn, w.num_q_heads, w.head_dim, device=dev, generator=gen) * scale).to(torch.bfloat16)
    dk = (torch.randn(b, dn, w.num_kv_heads, w.head_dim, device=dev, generator=gen) * scale).to(torch.bfloat16)
    dv = (torch.randn(b, dn, w.num_kv_heads, w.head_dim, device=dev, generator=gen) * scale).to(torch.bfloat16)
    dnn = torch.full((b,), dn, dtype=torch.int32, device=dev)
    dout = torch.zeros(b, dn, w.num_q_heads, w.head_dim, dtype=torch.bfloat16, device=dev)
    dws = torch.empty(T.tree_verify_attn_workspace_size((b, dn, w.num_q_heads, w.head_dim), cache,
                                                        p_max), dtype=torch.uint8, device=dev)

    def drafter_level():
        T.draft_grow_mask(dmask, dpos, last[1], prefix_t, last[0])
        T.tree_verify_attn(dq, dk, dv, cache, prefix_t, dnn, dpos, dmask, w.theta, sm_scale,
                           dout, dws, p_max)

    def sample_accept():
        T.tree_sample_accept(sa_logits, *sa_prm, sa_u, sa_uf, hp.tokens, hp.next_token,
                             hp.next_sibling, hp.num_nodes, prefix_t, shape.max_depth, cache,
                             *sa_out, sa_ws)

    def topk_level():  # one expansion level (level 2: [B, K, V] rows)
        T.draft_topk_expand(levels[1], k, 2, hp.front[0][1], hp.front[0][2], hp.store_token,
                            hp.store_score, hp.store_parent, *lvl_out, lvl_ws)

    legs = {"step": step, "attn": attn, "topk": topk_level, "lm_head": lm_head,
            "sample": sample_accept, "topk_product": topk_product, "variants": variants,
            "drafter": drafter_level}
    sides = {}
    if not args.no_side:
        for name, want in SIDE_LEGS:
            if name != w.name:
                sides[name] = side_state(name, want, dev, gen, T)
                legs.update(sides[name]["fns"])
                print(f"bench: side legs of {name} ready", file=sys.stderr, flush=True)

    def leg_bytes(name):
        """Algorithmic input bytes of one call of an attention or top-k leg (0 for the
        others, which are timed only one call at a time after a flush)."""
        if name == "attn":
            return algorithmic(w, prefix, depths)[0]
        if name == "topk":
            return b * k * v * 4
        for sname, sd in sides.items():
            if name == "attn_" + sname:
                return algorithmic(sd["w"], sd["prefix"], sd["depths"])[0]
            if name == "topk_" + sname:
                return sd["w"].batch * sd["w"].top_k * sd["w"].vocab * 4
        return 0
    chain_legs = [n for n in legs if leg_bytes(n) > L2_BYTES]

    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    graphs = {}
    with torch.cuda.stream(stream):
        for _ in range(2):  # warm the allocator and the kernels before capture
            for fn in legs.values():
                fn()
        stream.synchronize()
        for name, fn in legs.items():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            graphs[name] = g
        # A leg whose inputs exceed L2 is also timed as CHAIN calls back to back in one
        # graph (no flush between them: each call streams its inputs from HBM): the
        # per-call time inside a step, without the launch latency of a graph of one call.
        for name in chain_legs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(CHAIN):
                    legs[name]()
            graphs[name + "@chain"] = g
    torch.cuda.synchronize()

    def timed_loop(n, record):
        ev = {name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(n)] for name in graphs}
        with torch.cuda.stream(stream):
            for i in range(n):
                for name in graphs:
                    flush_buf.zero_()
                    ev[name][i][0].record(stream)
                    graphs[name].replay()
                    ev[name][i][1].record(stream)
        return ev

    timed_loop(args.warmup, False)
    torch.cuda.synchronize()
    if args.steps is None:
        # enough steps for about 2 s of timed work (so the clock samples fall inside it)
        t = time.perf_counter()
        timed_loop(5, False)
        torch.cuda.synchronize()
        per = (time.perf_counter() - t) / 5
        args.steps = int(max(50, min(20000, 2.0 / max(per, 1e-6))))
        # every rank times the same number of steps
        args.steps = int(max_over_ranks([args.steps], world)[0])
    if world > 1:
        dist.barrier()
    import tempfile
    clocks = Clocks(os.path.join(os.environ.get("TSV_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"tsv_clocks_rank{rank}.csv"))
    with clocks:
        torch.cuda.synchronize()
        clocks.start()
        t_wall = time.perf_counter()
        ev = timed_loop(args.steps, True)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        clocks.stop()
    if world > 1:
        dist.barrier()
    ms = {name: sum(a.elapsed_time(c) for a, c in ev[name]) / args.steps for name in ev}
    for name in chain_legs:  # per call
        ms[name + "@chain"] /= CHAIN
    print("bench: timed region done", file=sys.stderr, flush=True)

    # ---- end to end through host buffers --------------------------------------------
    pin = lambda t: t.cpu().pin_memory()
    h_levels = [pin(x) for x in levels]
    h_q, h_k, h_v, h_tgt, h_root = pin(q), pin(k_new), pin(v_new), pin(target_t), pin(root)
    h_out = {n: torch.empty_like(t, device="cpu").pin_memory() for n, t in
             (("len", hp.accept_len), ("path", hp.accept_path), ("bonus", hp.bonus),
              ("newlen", hp.new_prefix_len))}
    h2d = sum(x.numel() * x.element_size() for x in h_levels + [h_q, h_k, h_v, h_tgt, h_root])
    d2h = sum(x.numel() * x.element_size() for x in h_out.values())

    # The end-to-end step as one graph: the inputs cross from pinned host memory on a
    # copy stream, level by level, while the expansion of the levels already in place
    # runs; the results come back at the end. Every byte still crosses in every step.
    copy_stream = torch.cuda.Stream(device=dev)
    lev_ready = [torch.cuda.Event() for _ in levels]
    in_ready = torch.cuda.Event()

    def e2e_body():
        fork = torch.cuda.Event()
        fork.record(stream)
        copy_stream.wait_event(fork)
        with torch.cuda.stream(copy_stream):
            root.copy_(h_root, non_blocking=True)
            for src, dst, ev in zip(h_levels, levels, lev_ready):
                dst.copy_(src, non_blocking=True)
                ev.record(copy_stream)
            for src, dst in ((h_q, q), (h_k, k_new), (h_v, v_new), (h_tgt, target_t)):
                dst.copy_(src, non_blocking=True)
            in_ready.record(copy_stream)
        hp.step(levels, root, q, k_new, v_new, prefix_t, target_t, w.theta, sm_scale,
                level_ready=lev_ready, inputs_ready=in_ready)
        h_out["len"].copy_(hp.accept_len, non_blocking=True)
        h_out["path"].copy_(hp.accept_path, non_blocking=True)
        h_out["bonus"].copy_(hp.bonus, non_blocking=True)
        h_out["newlen"].copy_(hp.new_prefix_len, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_body()
        stream.synchronize()
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e, stream=stream):
            e2e_body()
    torch.cuda.synchronize()

    def e2e_once():
        g_e2e.replay()

    e2e_ms = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + min(args.steps, 200)):  # a sample of the timed steps
            flush_buf.zero_()
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_once()
            c.record(stream)
            c.synchronize()
            if i >= args.warmup:
                e2e_ms.append(a.elapsed_time(c))
    e2e_step_ms = sum(e2e_ms) / len(e2e_ms)
    print("bench: end-to-end leg done", file=sys.stderr, flush=True)

    # ---- max over ranks ---------------------------------------------------------------
    step_ms, e2e_step_ms = max_over_ranks([ms["step"], e2e_step_ms], world)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    hbm, tf, src = peaks()

    def us_of(name):
        """Per-call µs of a leg: the chained figure when its inputs exceed L2."""
        return (ms[name + "@chain"] if name in chain_legs else ms[name]) * 1e3

    def timing(name, roof):
        """How a roofline's time was taken, with the one-call figure beside a chain's."""
        if name in chain_legs:
            alone = ms[name] * 1e3
            roof["timing"] = (f"{CHAIN} calls back to back in one graph, per call (inputs "
                              f"larger than L2, no flush between them)")
            roof["us_per_launch_alone"] = alone
            roof["frac_alone"] = roof["frac"] * roof["us_per_launch"] / alone
        else:
            roof["timing"] = "one call in a graph of its own after a 256 MiB L2 flush"
        return roof
    attn_roof = timing("attn", attn_roofline(w, prefix, depths, us_of("attn"), hbm, tf, src))
    topk_roof = timing("topk", topk_roofline(w, us_of("topk"), hbm, src))
    attn_s = us_of("attn") / 1e6
    lm_s = ms["lm_head"] / 1e3
    lm_bytes = lm_v * lm_h * 2 + lm_rows * lm_h * 2 + lm_rows * 4
    lm_flops = 2 * lm_rows * lm_v * lm_h
    lm_bound = "hbm" if lm_bytes / (hbm * 1e9) >= lm_flops / (tf * 1e12) else "tensor"
    if lm_bound == "hbm":
        lm_ach, lm_peak, lm_unit = lm_bytes / lm_s / 1e9, hbm, "GB/s"
    else:
        lm_ach, lm_peak, lm_unit = lm_flops / lm_s / 1e12, tf, "TFLOP/s"
    lm_roof = {"kernel": f"lm_head_argmax (tcgen05 GEMM + argmax epilogue, {lm_rows} rows x "
                         f"{lm_v} vocab x {lm_h} hidden, bf16)",
               "bound": lm_bound, "achieved": lm_ach, "peak": lm_peak, "unit": lm_unit,
               "frac": lm_ach / lm_peak, "peak_source": src,
               "traffic": traffic("lm_head", w.name)[0],
               "traffic_source": traffic("lm_head", w.name)[1],
               "algorithmic_bytes": lm_bytes, "algorithmic_flops": lm_flops,
               "us_per_launch": ms["lm_head"] * 1e3}
    sa_s = ms["sample"] / 1e3
    sa_bytes = int(nodes.sum()) * sa_v * 4
    sa_gbps = sa_bytes / sa_s / 1e9
    sa_roof = {"kernel": f"tree_sample_accept (filter + rejection walk + compaction; "
                         f"{int(nodes.sum())} nodes x {sa_v} fp32 logits, T 0.8, top-p 0.9)",
               "bound": "hbm", "achieved": sa_gbps, "peak": hbm, "unit": "GB/s",
               "frac": sa_gbps / hbm, "peak_source": src,
               "traffic": traffic("sample", w.name)[0],
               "traffic_source": traffic("sample", w.name)[1],
               "algorithmic_bytes": sa_bytes, "us_per_launch": ms["sample"] * 1e3}
    # the dominant kernel of the step: the attention call or the depth + 1 top-k levels
    dominant = "topk" if us_of("topk") * (w.depth + 1) > us_of("attn") else "attn"
    kernels_step = hp.kernels_per_step()
    # one expansion level ([B, K, V] rows): one kernel, or two for a large batch
    lvl_launches = T.draft_topk_expand_launches(b, k, v, k)

    def side_launches(sd):
        sw = sd["w"]
        n = 0
        for leg in sd["fns"]:
            if leg.startswith("attn_"):
                n += sd["attn_launches"]
            else:
                n += T.draft_topk_expand_launches(sw.batch, sw.top_k, sw.vocab, sw.top_k)
        return n
    attn_kernels = hp.attn_kernels()

    def leg_launches(name):
        """Kernels of one call of an attention or top-k leg."""
        if name == "attn":
            return attn_kernels
        if name == "topk":
            return lvl_launches
        for sd in sides.values():
            if name in sd["fns"]:
                sw = sd["w"]
                return (sd["attn_launches"] if name.startswith("attn_") else
                        T.draft_topk_expand_launches(sw.batch, sw.top_k, sw.vocab, sw.top_k))
        return 0
    line = {
        "metric": METRIC, "value": world * 1e3 / step_ms, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded draft logits, q/k/v, KV cache; planted target argmax)",
        "config": {"workload": w.name, "batch": b, "prefix": (int(prefix.min()), int(prefix.max())),
                   "nodes": t_max, "top_k": k, "depth": w.depth, "vocab": v,
                   "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "paged": paged, "l2": ("flushed (256 MiB write) before every timed launch; legs whose inputs exceed "
                          f"L2 also timed as {CHAIN} calls in one graph"),
                   "parallelism": f"replicas x{world}", "graph": "CUDA graph per step"},
        "attn_us_per_layer": us_of("attn"),
        "attn_hbm_GBps": attn_roof["hbm_GBps"],
        "attn_roofline_us": attn_roof["roofline_us"],
        "topk_rows_per_s": topk_roof["rows_per_s"],
        "topk_hbm_GBps": topk_roof["achieved"],
        "nodes_kv_tokens_per_s": attn_roof["nodes_kv_tokens_per_s"],
        "roofline": topk_roof if dominant == "topk" else attn_roof,
        "roofline_attn": attn_roof,
        "roofline_topk": topk_roof,
        "lm_head_us": ms["lm_head"] * 1e3,
        "roofline_lm_head": lm_roof,
        "topk_product_us": ms["topk_product"] * 1e3,
        "topk_product_hbm_frac": topk_roof["algorithmic_bytes"] / (ms["topk_product"] / 1e3) / 1e9 / hbm,
        "d2t_map_plus_fixed_level_us": ms["variants"] * 1e3,
        "drafter_level_us": ms["drafter"] * 1e3,
        "drafter_nodes": dn,
        "drafter_attn_hbm_frac": algorithmic(w, prefix, [d_depth] * b)[0] / (ms["drafter"] / 1e3) / 1e9 / hbm,
        "sample_accept_us": ms["sample"] * 1e3,
        "roofline_sample_accept": sa_roof,
        "e2e": {"value": world * 1e3 / e2e_step_ms, "unit": UNIT, "ms_per_step": e2e_step_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        # timed region per iteration: the step graph, the attention call, one top-k level,
        # the lm-head argmax (GEMM + finalize), the non-greedy acceptance (filter, walk,
        # compaction), a product-score level, the d2t map and a fixed level, the drafter's
        # grown mask and its attention, the side legs, and the chained calls of the legs
        # whose inputs exceed L2
        "gpu_launches": args.steps * (kernels_step + attn_kernels + 2 * lvl_launches + 2 + 3 + 2 + 1 +
                                      T.tree_verify_attn_launches(
                                          (b, dn, w.num_q_heads, w.head_dim), cache, p_max) +
                                      sum(side_launches(sd) for sd in sides.values()) +
                                      CHAIN * sum(leg_launches(n) for n in chain_legs)),
        "wall_s_timed_region": t_wall,
    }
    for name, sd in sides.items():
        for leg in sd["fns"]:
            kind = leg.split("_")[0]
            if kind == "attn":
                line["roofline_attn_" + name] = timing(leg, attn_roofline(
                    sd["w"], sd["prefix"], sd["depths"], us_of(leg), hbm, tf, src))
            else:
                line["roofline_topk_" + name] = timing(leg, topk_roofline(
                    sd["w"], us_of(leg), hbm, src))
    ck = clocks.summary()
    if ck:
        line["clocks"] = ck
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(plain(line)))
    if world > 1:
        dist.destroy_process_group()


# --------------------------------------------------------------------------------------
def oracle_step_inputs(w, b):
    levels = [W.draft_logits(w, b, lvl) for lvl in range(1, w.depth + 2)]
    p = int(W.prefix_lengths(w)[b])
    q, k_new, v_new = W.new_qkv(w.with_(batch=b + 1))
    k_pre, v_pre = W.prefix_kv(w, b, p)
    return levels, p, q[b], k_new[b], v_new[b], k_pre, v_pre


def run_oracle_step(w, b, inputs):
    from oracle import step
    levels, p, q, k_new, v_new, k_pre, v_pre = inputs
    f64 = lambda x: np.asarray(x, np.float64)
    return step.hot_path_step(levels, w.top_k, w.total_tokens, int(W.root_tokens(w)[b]), f64(q),
                              f64(k_new), f64(v_new), f64(k_pre), f64(v_pre),
                              lambda t, par: W.plant_target(w, b, t, par), w.theta,
                              1 / math.sqrt(w.head_dim), w.depth + 2)


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


BLAS_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS",
            "BLIS_NUM_THREADS", "NUMEXPR_NUM_THREADS")


def _oracle_worker(job):
    """One process of a CPU leg (spawned with the BLAS thread variables at 1, so numpy
    runs on one thread): whole oracle steps of request `b` for `seconds`; returns
    (steps, seconds taken)."""
    name, b, seconds = job
    w = W.WORKLOADS[name]
    inputs = oracle_step_inputs(w, b)
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds or n == 0:
        run_oracle_step(w, b, inputs)
        n += 1
    return n, time.perf_counter() - t0


def _run_workers(name, seconds, workers, batch):
    """`workers` spawned processes, each on one BLAS thread, running oracle steps of
    independent requests at the same time; returns the per-worker (steps, seconds)."""
    import multiprocessing as mp
    saved = {k: os.environ.get(k) for k in BLAS_ENV}
    for k in BLAS_ENV:
        os.environ[k] = "1"  # read by numpy's BLAS when the spawned child imports it
    try:
        with mp.get_context("spawn").Pool(workers) as pool:
            return pool.map(_oracle_worker, [(name, i % batch, seconds) for i in range(workers)])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _mem_available_bytes():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def cpu_baseline(w, seconds):
    """The oracle timed on this host, in two legs of whole single-request oracle steps,
    each about `seconds` long: one thread (one spawned process on one BLAS thread), and
    all cores (one spawned process per core, each on one BLAS thread, independent
    requests). steps/s scaled to the workload's batch (a step processes all B
    requests). The all-core figure is `value`."""
    nproc = os.cpu_count() or 1
    # one thread: one spawned process
    (n, dt1), = _run_workers(w.name, seconds, 1, w.batch)
    one = 1.0 / (dt1 / n * w.batch)
    # all cores: as many workers as cores, fewer if host memory would not hold them
    per_worker = 3 << 30 if w.max_prefix > 8192 else 1 << 30
    avail = _mem_available_bytes()
    workers = nproc if avail is None else max(1, min(nproc, avail // per_worker))
    res = _run_workers(w.name, seconds, workers, w.batch)
    rate = sum(k / t for k, t in res)  # requests per second over all workers
    allc = rate / w.batch
    return {"value": allc, "unit": UNIT, "cores": int(workers), "kind": "oracle",
            "sample": f"{sum(k for k, _ in res)} single-request oracle steps of the {w.name} "
                      f"workload on {workers} processes (one BLAS thread each, about "
                      f"{seconds:.0f} s), scaled to a batch of {w.batch}",
            "one_thread": {"value": one, "unit": UNIT, "cores": 1,
                           "sample": f"{n} single-request oracle steps ({dt1:.1f} s) on one "
                                     f"thread, scaled to a batch of {w.batch}"},
            "nproc": nproc, "cpu_model": cpu_model()}


def reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload(args)
    if args.steps is None:
        args.steps = 3  # oracle steps take seconds: a small bounded sample
    inputs = [oracle_step_inputs(w, b) for b in range(min(w.batch, 2))]
    for i in range(args.warmup):
        run_oracle_step(w, i % len(inputs), inputs[i % len(inputs)])
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        run_oracle_step(w, i % len(inputs), inputs[i % len(inputs)])
        times.append(time.perf_counter() - t0)
    per_req = sum(times) / len(times)
    step_s = per_req * w.batch
    value = 1.0 / step_s
    line = {
        # n_gpus: the launch's N (the line the driver compares with); the oracle itself
        # runs on the host cores of rank 0
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": w.name, "batch": w.batch, "nodes": w.num_nodes,
                   "sample": "each timed step is one request's oracle step, scaled by batch"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"{args.steps} single-request oracle steps of {w.name}",
                         "nproc": os.cpu_count() or 1, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(plain(line)))


if __name__ == "__main__":
    a = parse()
    if a.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if a.impl == "reference":
        reference(a)
    else:
        native(a)
