"""Benchmark: sparse verification attention on one GB300 (or N replicas).

One step = one verification layer per layer of the workload through the
public per-layer call (sv_verify_layer): on a computing layer the fused
block scoring + budgeted top-k selection kernel, then the split-KV
tensor-core attention, which merges its partials in the same launch; on a
reuse layer (the 32-layer stack) only the attention, over the previous
computing layer's selection. Representatives are built at prefill and
rebuilt when a block fills (every blk / T steps), outside the step; that
update is timed on its own (`rep_update`).

Prints ONE JSON line (rank 0). Timing: W warm-up steps, then exactly K steps
replayed from CUDA graphs (one graph holding one step of every input set in
turn, so that consecutive steps chain as consecutive layers do, plus
single-step graphs for a remainder), bracketed by a barrier and a device
synchronize on both sides, CUDA events on the launching stream, max over
ranks. L2: the steps rotate over enough independent input sets that their
working set is >= 4x the L2 size, so every step reads cold HBM.

Roofline: the attention launch alone is timed with CUDA events on its stream
over a second loop of graph-replayed attention launches (rotating input sets,
at least 100 ms so the clock sampler sees it under load); algorithmic bytes
per launch are the selected K/V pages, the draft K/V, Q and O. The step's own
fraction (all algorithmic bytes of a step over the step time) is reported
beside it.

per_config: the same measurements, briefly, on the other workloads the
metric spans (32K, the 64K tree, the 32-layer stack); the tiny fp32 workload
is a parity case only.

--impl reference runs the CPU oracle (the only reference this method has) on
a bounded sample of the same workload and reports the same metric.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from sparse_verification_attention_gb300 import workloads as W  # noqa: E402

METRIC = "verify-attn draft tokens/s & achieved HBM GB/s (fraction of peak) at 32K-128K ctx"
UNIT = "draft tokens/s"
DEFAULT_WORKLOAD = "llama8b_128k_b4"


# --------------------------------------------------------------- byte model
def budget_k(wl: W.Workload) -> int:
    from sparse_verification_attention_gb300 import api
    return api.sv_budget_blocks(wl.budget, wl.ctx, wl.NB)


def attend_bytes(wl: W.Workload, k: int) -> int:
    """Algorithmic bytes of one attention launch (one layer)."""
    e = wl.elt
    sel_kv = wl.B * wl.Hkv * k * wl.blk * wl.d * e * 2
    draft = wl.B * wl.T * wl.Hkv * wl.d * e * 2
    q = o = wl.B * wl.T * wl.Hq * wl.d * e
    return sel_kv + draft + q + o


def layer_bytes(wl: W.Workload, k: int, computing: bool) -> int:
    """Algorithmic bytes of one layer of the step (one verification layer:
    the fp32 representative stream when the layer computes its selection,
    and the attention launch). Representatives are built at prefill and
    updated when a block fills, outside the step (timed separately)."""
    reps = wl.B * wl.Hkv * wl.NB * wl.d * 4 if computing else 0
    return reps + attend_bytes(wl, k)


def rep_update_bytes(wl: W.Workload) -> int:
    """One block's rep per (sequence, kv head): read its keys, write its rep."""
    return wl.B * wl.Hkv * (wl.blk * wl.d * wl.elt + wl.d * 4)


def step_bytes(wl: W.Workload, k: int) -> int:
    return sum(layer_bytes(wl, k, l % wl.compute_every == 0) for l in range(wl.layers))


# --------------------------------------------------------------- helpers
def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def attend_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("attend_tc.cu", "attend_fast.cu", "attend_generic.cu", "tc.h", "ptx.h",
              "internal.h"):
        with open(os.path.join(ROOT, "sparse_verification_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profile(wl_name: str):
    """ncu DRAM bytes per attention launch recorded under profiles/, or None
    when absent or taken on a different attention source."""
    p = os.path.join(ROOT, "profiles", "attend_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(wl_name)
    if not ent or ent.get("source_hash") != attend_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = f"/tmp/sva_clocks_{os.getpid()}.csv"

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) < 6:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[2:6]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


_T0 = time.perf_counter()


def log(msg: str):
    print(f"[bench {time.perf_counter() - _T0:7.1f}s] {msg}", file=sys.stderr, flush=True)


def check_status(sets, where: str):
    """Raise if any kernel of the bench raised a device-side status flag."""
    from sparse_verification_attention_gb300 import api
    for ss in sets:
        for st in ss.layers:
            flags = api.sv_read_status(st.ws)
            if flags:
                words = st.ws[:8].view(torch.int32).tolist()
                raise RuntimeError(f"device status flags {flags:#x} after {where} (words {words})")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world):
    if world > 1:
        import torch.distributed as dist
        # harness-only collectives (barrier, max of timings) on CPU tensors;
        # the data path has no collective
        dist.init_process_group("gloo")
        return dist
    return None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------- oracle arm
class OracleSample:
    """The CPU oracle on a bounded sample of the workload: sequence 0 of layer
    0, one (sequence, kv head) verification (score, budget, select, attend)
    per unit, rotating over the kv heads; representatives prebuilt (prefill,
    untimed). One unit is 1/(B*Hkv*layers) of a step, i.e. T/(Hkv*layers)
    draft tokens' worth of verification."""

    def __init__(self, wl: W.Workload, x_cpu=None):
        from oracle import sva_oracle as O
        self.O, self.wl = O, wl
        if x_cpu is None:
            x_cpu = W.make_layer(W.scaled(wl, layers=1) if wl.layers > 1 else wl, 0, device="cpu")
        pages = x_cpu.block_table[0].long()
        self.kp = x_cpu.k_pool[pages].contiguous()
        self.vp = x_cpu.v_pool[pages].contiguous()
        self.bt = torch.arange(wl.NB, dtype=torch.int32).view(1, -1)
        self.q, self.dk, self.dv = x_cpu.q[:1], x_cpu.draft_k[:1], x_cpu.draft_v[:1]
        self.reps = O.block_representatives(self.kp, self.bt, wl.NB, wl.blk)
        self.i = 0

    def unit(self):
        wl, h = self.wl, self.i % self.wl.Hkv
        self.i += 1
        G = wl.G
        self.O.verify_layer(self.q[:, :, h * G:(h + 1) * G], self.kp[:, h:h + 1],
                            self.vp[:, h:h + 1], self.bt, self.dk[:, :, h:h + 1],
                            self.dv[:, :, h:h + 1], wl.parent_list(), wl.ctx, wl.blk, wl.budget,
                            reps=self.reps[:, h:h + 1])

    def tokens_per_unit(self) -> float:
        # a step is B*Hkv*layers such units for B*T draft tokens
        return self.wl.T / (self.wl.Hkv * self.wl.layers)

    def timed(self, seconds: float = 0.0, units: int = 0):
        n, t0 = 0, time.perf_counter()
        while True:
            self.unit()
            n += 1
            el = time.perf_counter() - t0
            if (units and n >= units) or (not units and el >= seconds):
                break
        return n, el

    def describe(self, n, el) -> str:
        return (f"{n} (sequence, kv head) verifications of sequence 0, layer 0 of {self.wl.name} "
                f"(score {self.wl.NB} reps, budget, top-k, attend), {el:.1f} s of CPU time, "
                f"fp64 PyTorch-CPU oracle")


def run_reference(args, wl, rank, world):
    if rank != 0:
        return
    o = OracleSample(wl)
    o.timed(units=1)
    t_unit = o.timed(units=2)[1] / 2
    # size each step so that warm-up + K steps stay within about two minutes
    per_step = max(1, min(wl.Hkv, int(120.0 / max(1, args.steps + args.warmup) / t_unit)))
    o.timed(units=per_step * args.warmup)
    n, el = o.timed(units=per_step * args.steps)
    tok_s = n * o.tokens_per_unit() / el
    desc = o.describe(n, el) + f"; {per_step} per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": tok_s, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(wl, o.O.budget_from(wl.budget, wl.ctx, wl.NB)),
        "cpu_baseline": {"value": tok_s, "unit": UNIT, "cores": os.cpu_count(),
                         "threads": torch.get_num_threads(), "kind": "oracle", "sample": desc},
        "e2e": {"value": tok_s, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(wl: W.Workload, k):
    return {"workload": f"{wl.name}: {wl.description}", "B": wl.B, "ctx": wl.ctx, "T": wl.T,
            "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d, "blk": wl.blk, "layers": wl.layers,
            "budget_blocks": k, "draft_mask": "chain" if wl.parents is None else
            "tree " + ",".join(map(str, wl.parents)), "parallelism": "replicas (1 GPU each)"}


# --------------------------------------------------------------- GPU arm
class StepSet:
    """One independent input set resident in HBM (one per layer of a stack)."""

    def __init__(self, wl, index, layers_planted):
        from sparse_verification_attention_gb300 import api
        self.layers = []
        for l in range(wl.layers):
            x = W.make_layer(wl, index * wl.layers + l, device="cuda",
                             planted=layers_planted[l])
            self.layers.append(api.LayerState(wl, x))
        # reuse layers share the computing layer's selection slot
        for l in range(wl.layers):
            if l % wl.compute_every:
                self.layers[l].slot = self.layers[l - (l % wl.compute_every)].slot


def run_step(wl, ss: StepSet):
    """Launch one step on the current stream (graph-capturable): one
    sv_verify_layer call per layer, computing or reusing the selection."""
    from sparse_verification_attention_gb300 import api
    for l, st in enumerate(ss.layers):
        reuse = api.VERIFY_COMPUTE if l % wl.compute_every == 0 else api.VERIFY_REUSE
        api.sv_verify_layer(st.shape, st.x.q, st.kv, st.reps, wl.budget, st.x.draft_k,
                            st.x.draft_v, st.parents, reuse, st.slot, st.out, st.ws)


def attend_launch(st):
    """The attention of one layer alone, over the layer's own selection."""
    from sparse_verification_attention_gb300 import api
    api.sv_sparse_attend(st.shape, st.x.q, st.kv, st.sel, st.k, st.kmax, st.x.draft_k,
                         st.x.draft_v, st.parents, st.out, st.ws)


def timed_replays(graph_fn, min_ms: float, per_replay_units: int):
    """Replay a graph until at least min_ms of device time (after one
    untimed replay); returns ms per unit. CUDA events on the current stream."""
    graph_fn()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    graph_fn()
    a1.record()
    torch.cuda.synchronize()
    once = max(a0.elapsed_time(a1), 1e-3)
    n = max(3, int(math.ceil(min_ms / once)))
    a0.record()
    for _ in range(n):
        graph_fn()
    a1.record()
    torch.cuda.synchronize()
    return a0.elapsed_time(a1) / (n * per_replay_units)


def sdpa_dense(wl, st):
    """torch SDPA over the whole context gathered into logical order, with the
    draft mask (a dense yardstick from a library kernel; the gather is done
    once, outside the timing). Returns ms per call, or a reason string."""
    import torch.nn.functional as F
    x = st.x
    try:
        nbt = wl.NBT
        pages = x.block_table[:, :nbt].long()                              # [B, nbt]
        def ctx_of(pool):
            g = pool[pages]                                                # [B, nbt, Hkv, blk, d]
            g = g.permute(0, 2, 1, 3, 4).reshape(wl.B, wl.Hkv, nbt * wl.blk, wl.d)
            return g[:, :, :wl.ctx]
        k = torch.cat([ctx_of(x.k_pool), x.draft_k.transpose(1, 2)], dim=2).contiguous()
        v = torch.cat([ctx_of(x.v_pool), x.draft_v.transpose(1, 2)], dim=2).contiguous()
        q = x.q.transpose(1, 2).contiguous()                               # [B, Hq, T, d]
        mask = torch.zeros(wl.T, wl.ctx + wl.T, dtype=torch.bool, device=q.device)
        mask[:, :wl.ctx] = True
        par = wl.parent_list()
        for t in range(wl.T):
            u = t
            while u >= 0:
                mask[t, wl.ctx + u] = True
                u = par[u]
        call = lambda: F.scaled_dot_product_attention(q, k, v, attn_mask=mask, enable_gqa=True)
        call()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(5)]
        for a, b in ev:
            a.record()
            call()
            b.record()
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        del k, v, q
        torch.cuda.empty_cache()
        return ms
    except (RuntimeError, TypeError) as e:  # backend without this mask/GQA form
        return f"unavailable: {str(e).splitlines()[0][:160]}"


def measure(args, wl, dist, steps: int, warmup: int, full: bool, clocks=None):
    """Every GPU number of one workload: the timed steps, the attention
    roofline loop, the e2e loop; with full=True also the dense yardsticks and
    the rep update. Returns (fields, sets, k)."""
    from sparse_verification_attention_gb300 import api
    k = budget_k(wl)
    sbytes = step_bytes(wl, k)
    abytes = attend_bytes(wl, k)
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = getattr(props, "L2_cache_size", 129 * 2 ** 20)
    n_sets = max(2, math.ceil(4 * l2 / sbytes))
    if args.sets:
        n_sets = args.sets
    ps = W.planted_sets(wl)
    sets = [StepSet(wl, i, ps) for i in range(n_sets)]
    torch.cuda.synchronize()
    log(f"{wl.name}: {n_sets} input sets resident")
    stream = torch.cuda.current_stream()

    # one CUDA graph per input set, each holding one whole step
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for ss in sets:  # warm the launch paths once outside capture
            run_step(wl, ss)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graphs = []
    for ss in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run_step(wl, ss)
        graphs.append(g)
    # one step of every set in turn in one graph: consecutive steps chain as
    # consecutive layers do (each kernel's dependents launch early and wait
    # on it), which separate graph launches would not
    rotation = torch.cuda.CUDAGraph()
    with torch.cuda.graph(rotation):
        for ss in sets:
            run_step(wl, ss)
    torch.cuda.synchronize()
    check_status(sets, "graph capture")

    def replay_steps(n):  # exactly n steps: whole rotations, then single steps
        for _ in range(n // n_sets):
            rotation.replay()
        for i in range(n % n_sets):
            graphs[i].replay()

    if clocks is not None:
        clocks.start()
    replay_steps(warmup)
    barrier(dist)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    replay_steps(steps)
    e1.record()
    torch.cuda.synchronize()
    barrier(dist)
    ms_total = max_over_ranks(dist, e0.elapsed_time(e1))
    check_status(sets, "timed steps")
    ms_step = ms_total / steps
    tokens = sum_over_ranks(dist, wl.B * wl.T * steps)
    log(f"{wl.name}: timed steps {ms_step * 1e3:.1f} us/step")

    # roofline: the attention launches alone, back to back as in a layer
    # stack, one CUDA graph of kRoofLaunches launches rotating over the input
    # sets (cold L2), replayed for at least 100 ms; CUDA events on the stream
    kRoofLaunches = 20
    att_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(att_graph):
        for i in range(kRoofLaunches):
            for st in sets[i % n_sets].layers:
                attend_launch(st)
    attend_ms = timed_replays(att_graph.replay, 100.0 if full else 20.0,
                              kRoofLaunches * wl.layers)
    if clocks is not None:
        clk = clocks.stop()
    else:
        clk = None
    check_status(sets, "attention-only replays")
    log(f"{wl.name}: attention launches {attend_ms * 1e3:.1f} us")
    peak, peak_kind = read_peaks()
    achieved = abytes / (attend_ms / 1e3) / 1e9
    step_gbs = sbytes / (ms_step / 1e3) / 1e9
    st0 = sets[0].layers[0]
    plan = api.sv_attend_plan(st0.shape, st0.kv, k)
    f = {
        "value": tokens / (ms_total / 1e3), "ms_per_step": ms_step, "k": k,
        "n_sets": n_sets, "l2": l2, "step_bytes": sbytes, "step_gbs": step_gbs,
        "step_frac": step_gbs / peak, "attend_bytes": abytes, "attend_ms": attend_ms,
        "attend_gbs": achieved, "attend_frac": achieved / peak, "peak": peak,
        "peak_kind": peak_kind, "plan": plan, "clocks": clk,
    }

    if full and args.dense and wl.NB:
        # dense full-KV verification: the same kernels with every block kept,
        # and torch SDPA over the gathered context
        dws = api.alloc_workspace(st0.shape, wl.NB, wl.NB)
        dout = torch.empty_like(st0.out)
        dcall = lambda: api.sv_sparse_attend(st0.shape, st0.x.q, st0.kv, None, 0, 0,
                                             st0.x.draft_k, st0.x.draft_v, st0.parents, dout, dws)
        dcall()
        de = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(5)]
        for a, b in de:
            a.record()
            dcall()
            b.record()
        torch.cuda.synchronize()
        dms = statistics.median(a.elapsed_time(b) for a, b in de)
        dbytes = attend_bytes(wl, wl.NB)
        sd = sdpa_dense(wl, st0)
        f["dense"] = {"attend_ms": dms, "gbs": dbytes / (dms / 1e3) / 1e9,
                      "sparse_speedup": dms / attend_ms, "note": "same kernels, all blocks kept",
                      "torch_sdpa_ms": sd if isinstance(sd, float) else None,
                      "torch_sdpa_note": ("torch scaled_dot_product_attention over the "
                                          "gathered context + drafts with the draft mask, GQA"
                                          if isinstance(sd, float) else sd),
                      "sparse_speedup_vs_sdpa": (sd / attend_ms) if isinstance(sd, float) else None}
        del dws, dout

    if full and wl.NB:
        # the incremental rep update (one newly filled block per (b, h)),
        # outside the step: a block fills every blk / T steps
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(kRoofLaunches):
                st = sets[i % n_sets].layers[0]
                api.sv_build_reps(st.shape, st.kv, wl.NB - 1, 1, st.reps)
        rms = timed_replays(g.replay, 5.0, kRoofLaunches)
        f["rep_update"] = {"us_per_layer": rms * 1e3, "bytes_per_layer": rep_update_bytes(wl),
                           "every_steps": wl.blk / max(1, wl.T),
                           "note": "sv_build_reps of one newly filled block per (b, h); "
                                   "not in the step"}

    # e2e: the public call with host buffers, copies inside the timed region
    f["e2e"] = run_e2e(args, wl, sets, dist)
    check_status(sets, "e2e")
    f["launches_per_step"] = sum((1 if l % wl.compute_every == 0 else 0) +
                                 (1 if (plan.path == api.SV_PATH_TCGEN05 or plan.cluster > 0)
                                  else 2) for l in range(wl.layers))
    return f, sets, k


def run_gpu(args, wl, rank, world, dist):
    from sparse_verification_attention_gb300 import api, build_lib
    build_lib.build()
    dev = args.local_rank
    torch.cuda.set_device(dev)
    clocks = ClockSampler(dev)
    f, sets, k = measure(args, wl, dist, args.steps, args.warmup, True, clocks)
    log("headline done")

    # CPU oracle baseline on a bounded sample (rank 0, N=1 only): all host
    # cores, and one thread
    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        o = OracleSample(wl, sets[0].layers[0].x.to("cpu"))
        n, el = o.timed(seconds=args.cpu_seconds)
        threads = torch.get_num_threads()
        torch.set_num_threads(1)
        try:
            n1, el1 = o.timed(seconds=max(2.0, args.cpu_seconds / 3))
        finally:
            torch.set_num_threads(threads)
        cpu = {"value": n * o.tokens_per_unit() / el, "unit": UNIT, "cores": os.cpu_count(),
               "threads": threads, "kind": "oracle", "sample": o.describe(n, el),
               "single_thread": {"value": n1 * o.tokens_per_unit() / el1, "unit": UNIT,
                                 "sample": o.describe(n1, el1)}}
    del sets
    torch.cuda.empty_cache()

    # the other workloads of the metric's range, briefly (the same kernels,
    # the same measurements; no dense yardsticks)
    per_config = {}
    if args.per_config:
        for name in ("llama8b_32k", "qwen3moe_64k_b8_tree16", "llama8b_60k_32layer"):
            if name == wl.name:
                continue
            owl = W.WORKLOADS[name]
            of, osets, ok_ = measure(args, owl, dist, args.per_config_steps, 3, False)
            del osets
            torch.cuda.empty_cache()
            per_config[name] = {
                "metric": METRIC, "unit": UNIT, "value": of["value"],
                "ms_per_step": of["ms_per_step"], "budget_blocks": ok_,
                "step_bytes": of["step_bytes"], "step_frac": of["step_frac"],
                "attend_us": of["attend_ms"] * 1e3, "attend_frac": of["attend_frac"],
                "attend_bytes": of["attend_bytes"],
                "attend_traffic": traffic_from_profile(owl.name),  # ncu DRAM bytes, or None
                "e2e": {"value": of["e2e"]["value"], "ms_per_step": of["e2e"]["ms_per_step"]},
                "config": config_of(owl, ok_)}
        per_config["tiny_f32"] = {"parity_only": True,
                                  "note": "oracle-sized fp32 case; checked element by element "
                                          "in the GPU tests, not timed"}

    traffic = traffic_from_profile(wl.name)
    plan = f["plan"]
    line = {
        "metric": METRIC, "value": f["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": f["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded Gaussian Q/K/V, planted high-affinity blocks + sink)",
        "config": dict(config_of(wl, k), l2=(
            f"rotating {f['n_sets']} input sets, {f['n_sets'] * f['step_bytes'] / 1e6:.0f} MB "
            f"touched per rotation vs {f['l2'] / 1e6:.0f} MB L2 (inputs larger than L2, "
            f"no flush)")),
        "step_bytes": f["step_bytes"], "step_gbs": f["step_gbs"],
        "step_frac": f["step_frac"],
        "roofline": {"bound": "hbm", "achieved": f["attend_gbs"], "peak": f["peak"],
                     "unit": "GB/s", "frac": f["attend_frac"], "traffic": traffic,
                     "kernel": {api.SV_PATH_TCGEN05: "attend_tc_kernel (tcgen05 split-KV "
                                "attention, LSE merge in the same launch: "
                                + ("through distributed shared memory, one cluster per pair"
                                   if plan.cluster else "by the CTA holding each pair's last "
                                   "ticket") + ")",
                                api.SV_PATH_MMA_SYNC: "attend_fast_kernel (mma.sync split-KV)",
                                api.SV_PATH_CUDA_CORES: "attend_generic_kernel + merge_kernel"
                                }[plan.path],
                     "bytes_per_launch": f["attend_bytes"], "launch_ms": f["attend_ms"],
                     "peak_kind": f"{f['peak_kind']} HBM copy bandwidth (burst)",
                     "frac_of_nominal_8tbs": f["attend_gbs"] / 8000.0,
                     "step_frac": f["step_frac"],
                     "step_frac_of_nominal_8tbs": f["step_gbs"] / 8000.0},
        "dense": f.get("dense"),
        "rep_update": f.get("rep_update"),
        "e2e": f["e2e"],
        "cpu_baseline": cpu,
        "per_config": per_config or None,
        "gpu_launches": f["launches_per_step"] * args.steps,
        "clocks": f["clocks"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, wl, sets, dist):
    """sv_verify_layer_host per layer: the public call with the step's
    per-token inputs (Q, draft K, draft V) in pinned host memory and the
    output copied back to host memory, all inside the timed region. The
    library runs the input copies on one copy stream and the output copy on
    another, ordered against the compute stream by events, so a step's copies
    overlap the neighbouring steps' kernels. Steps rotate over the same input
    sets as the device-timed loop; a set's device buffers are refilled only
    after the step that last used them has been copied back."""
    from sparse_verification_attention_gb300 import api
    host = []
    for ss in sets:
        host.append([(st.x.q.cpu().pin_memory(), st.x.draft_k.cpu().pin_memory(),
                      st.x.draft_v.cpu().pin_memory(),
                      torch.empty_like(st.out, device="cpu").pin_memory()) for st in ss.layers])
    h2d = sum(t.numel() * t.element_size() for hq, hk, hv, _ in host[0] for t in (hq, hk, hv))
    d2h = sum(ho.numel() * ho.element_size() for *_, ho in host[0])
    steps = max(3, min(args.steps, args.e2e_steps))
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    S = len(sets)
    done = [torch.cuda.Event() for _ in range(S)]
    used = [False] * S

    def one(i):
        j = i % S
        ss, hb = sets[j], host[j]
        if used[j]:
            cin.wait_event(done[j])  # this set's last output has been read back
        for l, st in enumerate(ss.layers):
            hq, hk, hv, ho = hb[l]
            reuse = int(l % wl.compute_every != 0)
            api.sv_verify_layer_host(st.shape, hq, st.x.q, st.kv, st.reps, wl.budget, hk, hv,
                                     st.x.draft_k, st.x.draft_v, st.parents, reuse, st.slot, ho,
                                     st.out, st.ws, comp, cin, cout)
        done[j].record(cout)
        used[j] = True

    for i in range(3):
        one(i)
    comp.wait_stream(cout)
    barrier(dist)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    cin.wait_stream(comp)  # the first copies start inside the timed region
    for i in range(steps):
        one(i)
    comp.wait_stream(cout)  # the last output is on the host
    e1.record(comp)
    torch.cuda.synchronize()
    barrier(dist)
    ms = max_over_ranks(dist, e0.elapsed_time(e1))
    tokens = sum_over_ranks(dist, wl.B * wl.T * steps)
    return {"value": tokens / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps,
            "note": "sv_verify_layer_host per layer (host buffers; input and output copies on "
                    "their own streams), rotating input sets"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--sets", type=int, default=0)
    ap.add_argument("--dense", type=int, default=1)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--per-config", type=int, default=1)
    ap.add_argument("--per-config-steps", type=int, default=200)
    args = ap.parse_args()
    rank, world, local = dist_env()
    args.local_rank = local
    wl = W.WORKLOADS[args.workload]
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args, wl, rank, world)
        return
    dist = init_dist(world)
    try:
        run_gpu(args, wl, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
