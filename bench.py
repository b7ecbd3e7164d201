"""Benchmark: verified draft tokens/s through 30 GDN layers of verify + accept + rollback.

One step = one speculative round of the workload: gdn_verify over all layers (one launch),
spec_accept over the verify logits, gdn_rollback over all layers (one launch). Inputs are seeded
synthetic tensors with the workload's shapes, resident in HBM before timing (a pool of rounds is
cycled); the recurrent state (4 GB for the batched workload) is far larger than L2, so every step
streams it from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 2]

Prints one JSON line (rank 0). Under torchrun each rank runs its own copy of the workload on its
own GPU (weak scaling; sequences are independent, so there is no collective on the data path).
--impl reference times the CPU oracle on the host cores on the same workload and metric.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified draft tokens/sec (30 GDN layers+accept+rollback); % HBM roofline"
UNIT = "tokens/s"
DEFAULT_CONFIG = 2
POOL = 4


# ------------------------------------------------------------------------------ distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return ws, rank


def rank_seed(seed, rank):
    """Each rank draws its own sequences (weak scaling): distinct, reproducible seeds."""
    return int(seed) * 1000003 + int(rank)


def reduce_max(x, device=None):
    """Max of a float over ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate_tokens_per_s(world, B, N, ms_per_step):
    return world * B * N / (ms_per_step / 1e3)


# ------------------------------------------------------------------------------ accounting
def gate_bytes(w):
    """Bytes of one position's gates: one fp32 per value head, or one per key channel."""
    return 4 * w.Hv * (w.D if getattr(w, "gate_dk", False) else 1)


def bytes_verify(w):
    """Algorithmic HBM bytes of one gdn_verify launch over the whole workload: each input read
    once, each output written once (state S_0 read, never written)."""
    io = 2 if str(w.io_dtype).endswith("bfloat16") else 4
    S = w.Hv * w.D * w.D * 4
    T, C = w.N, w.C
    per_unit = (S + T * (io * C + 4 * w.Hv + gate_bytes(w) + io * w.Hv * w.D + 4 * w.Hv * w.D
                         + 4 * w.Hk * w.D)
                + io * (w.W - 1) * C)
    return w.L * w.B * per_unit + w.L * io * C * w.W


def bytes_rollback(w, n_list):
    """Algorithmic bytes of one gdn_rollback launch for accepted counts n_list (one per seq)."""
    io = 2 if str(w.io_dtype).endswith("bfloat16") else 4
    S = w.Hv * w.D * w.D * 4
    C, W = w.C, w.W
    tot = 0
    for n in n_list:
        n = int(n)
        if n <= 0:
            continue
        m = min(n, W - 1)
        tot += (2 * S + n * (4 * w.Hv * w.D + 4 * w.Hk * w.D + gate_bytes(w))
                + io * (W - 1 - m) * C + io * m * C + io * (W - 1) * C)
    return w.L * tot + 4 * w.B


def bytes_rollback_verify(w, n_list):
    """Algorithmic bytes of one gdn_rollback_verify launch: the verify's bytes (state read once)
    plus, for every (layer, sequence) with n > 0, the committed state written back, the previous
    tape read (δ, k, gates) and the conv window's previous rows read and the new conv rows
    written."""
    io = 2 if str(w.io_dtype).endswith("bfloat16") else 4
    S = w.Hv * w.D * w.D * 4
    C, W = w.C, w.W
    tot = 0
    for n in n_list:
        n = int(n)
        if n <= 0:
            continue
        tot += S + n * (4 * w.Hv * w.D + 4 * w.Hk * w.D + gate_bytes(w)) + 2 * io * (W - 1) * C
    return bytes_verify(w) + w.L * tot + 4 * w.B


def bytes_accept(w, n_list):
    """Algorithmic bytes of one accept call: the logits rows the accept loop reaches, n + 1 per
    sequence for n accepted drafts (rows 0..n: the judged drafts and the row of the correction,
    resample or bonus), plus the drafts read and the tokens and counts written. The greedy kernels
    read all N + 1 rows in parallel; the sampling kernel reads only the rows it reaches (and
    prefetches one more)."""
    io = 2 if str(w.io_dtype).endswith("bfloat16") else 4
    rows = sum(int(n) + 1 for n in n_list)
    return rows * w.V * io + 4 * w.B * (2 * w.N + 2)


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# the sources each timed kernel is built from (its counters go stale when one of them changes)
KERNEL_SOURCES = {
    "gdn_verify": ("verify_pipe.cuh", "verify_impl.cuh", "verify_bf16.cu", "tc.cuh", "common.cuh",
                   "kernels.h"),
    "gdn_rollback_verify": ("verify_pipe.cuh", "verify_impl.cuh", "verify_bf16.cu", "tc.cuh",
                            "common.cuh", "kernels.h"),
    "gdn_rollback": ("rollback.cu", "common.cuh", "kernels.h"),
    "spec_accept": ("accept.cu", "common.cuh", "kernels.h"),
    "attn_verify": ("attn.cu", "attn.h", "tc.cuh", "common.cuh"),
}


def kernel_sources_sha(kernel=None):
    """Hash of a kernel's sources (all of csrc when kernel is None): profile counters are stale
    once this changes."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_verify_gdn_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel) if kernel else None
    for name in sorted(names or os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def full_size(args):
    """Whether the run is the named workload itself (no --batch / --layers override): the
    profiled traffic records are per launch of the full workload."""
    return getattr(args, "batch", None) is None and getattr(args, "layers", None) is None


def profiled_traffic(workload_name, kernel):
    """dram read+write bytes per launch from a committed ncu summary, if it matches the sources."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload_name, {}).get(kernel)
        if e and e.get("src_sha") == kernel_sources_sha(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        return None
    return None


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ CPU oracle leg
def host_cores():
    """Host cores this process may run on (the affinity mask, else the CPU count)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_unit_times(w, seed, budget_s, units_min, threads=1):
    """Time the CPU oracle on (layer, sequence) units of verify+rollback and on per-sequence
    accepts of the workload, with `threads` oracle threads: each call covers one sequence per
    thread, and the times are per unit / per sequence of that throughput. Returns (seconds per
    unit, seconds per accepted sequence, units, threads in effect)."""
    import numpy as np
    import torch
    import oracle
    from speculative_verify_gdn_gb300 import inputs as I

    threads = oracle.set_threads(threads)
    try:
        nb = threads
        small = I.custom(w, name=w.name, L=1, B=nb)
        cw = I.model_weights(small, seed).double().numpy()
        st, cs = I.initial_state(small, seed)
        st, cs = st.double().numpy(), cs.double().numpy()
        qkv, g, beta = I.round_stream(small, 0, seed)
        qkv, g, beta = qkv.double().numpy(), g.double().numpy(), beta.double().numpy()
        d = oracle.OracleDims(L=1, B=nb, T=w.N, Hk=w.Hk, Hv=w.Hv, Dk=w.D, Dv=w.D, W=w.W)
        parent = None
        if w.accept == "tree":
            parent = np.tile(I.random_tree(I.custom(w, name=w.name, B=1), 0, seed).numpy(), (nb, 1))
        n = np.full(nb, max(1, w.N // 2), np.int32)
        path = None
        if parent is not None:
            path = np.full((nb, w.P), -1, np.int32)
            x, k = 0, 0
            while x >= 0 and k < n[0]:
                path[:, k] = x
                k += 1
                ch = [v for v in range(w.N) if parent[0, v] == x]
                x = ch[0] if ch else -1
            n[:] = k
        t0 = time.perf_counter()
        units = 0
        while units < units_min or time.perf_counter() - t0 < budget_s:
            ref = oracle.verify(d, qkv, cw, cs, g, beta, st, parent=parent)
            oracle.rollback(d, n, ref["tape_delta"], ref["tape_k"], g, qkv, st, cs, path=path)
            units += nb
        t_unit = (time.perf_counter() - t0) / units
        # accept: one sequence's N+1 rows per thread
        one = I.custom(w, name=w.name, B=nb)
        if w.accept == "sample":
            lg, dr = I.sample_logits(one, 0, seed)
        elif w.accept == "tree":
            par = I.random_tree(one, 0, seed)
            tok, lg, _ = I.tree_tokens_and_logits(one, par, 0, seed)
        else:
            lg, dr, _ = I.greedy_logits(one, 0, seed)
        lgf = lg.float().numpy()
        reps = 0
        t1 = time.perf_counter()
        while reps < 2 or time.perf_counter() - t1 < min(2.0, budget_s / 5):
            if w.accept == "sample":
                oracle.accept_sample(lgf, dr.numpy(), w.temperature, seed, reps)
            elif w.accept == "tree":
                oracle.accept_tree(lgf, par.numpy(), tok.numpy(), w.P)
            else:
                oracle.accept_greedy(lgf, dr.numpy())
            reps += 1
        t_acc = (time.perf_counter() - t1) / (reps * nb)
    finally:
        oracle.set_threads(1)
    del torch
    return t_unit, t_acc, units, threads


def cpu_tokens_per_s(w, t_unit, t_acc):
    """A sequence-round is L units of verify+rollback and one accept; it verifies N tokens."""
    return w.N / (w.L * t_unit + t_acc)


# ------------------------------------------------------------------------------ GPU leg
def workload_description(w):
    d = {"workload": "%s: %d GDN layers (Qwen3.6-shaped: Hk=%d, Hv=%d, d=%d, conv %d over C=%d), "
                     "batch %d, N=%d, %s accept over V=%d" % (
                         w.name, w.L, w.Hk, w.Hv, w.D, w.W, w.C, w.B, w.N, w.accept, w.V),
         "layers": w.L, "batch": w.B, "drafts": w.N, "vocab": w.V, "accept": w.accept,
         "io_dtype": "bf16" if str(w.io_dtype).endswith("bfloat16") else "f32",
         "state": "fp32 128x128 per value head, row-major S",
         "l2": "inputs larger than L2: the %.2f GB recurrent state is streamed from HBM every step"
               % (w.L * w.B * w.Hv * w.D * w.D * 4 / 1e9)}
    if getattr(w, "gate_dk", False):
        d["gates"] = "one decay per key channel, g [L, B, T, Hv, d]"
    if w.accept in ("greedy", "tree"):
        d["alphas"] = list(w.alphas)
    if w.accept == "sample":
        d["temperature"] = w.temperature
    if w.accept == "tree":
        d["tree"] = {"nodes": w.N, "depth": w.tree_depth, "branching": w.tree_branch}
    return d


def make_pool(w, seed, device, pool):
    import torch
    from speculative_verify_gdn_gb300 import inputs as I
    slots = []
    for k in range(pool):
        qkv, g, beta = I.round_stream(w, k, seed, device)
        parent = None
        if w.accept == "tree":
            par = I.random_tree(w, k, seed)
            tok, lg, _ = I.tree_tokens_and_logits(w, par, k, seed)
            parent, drafts, lg = par.to(device), tok.to(device), lg.to(device)
        elif w.accept == "sample":
            lg, drafts = I.sample_logits(w, k, seed, device)
        else:
            lg, drafts, _ = I.greedy_logits(w, k, seed, device)
        slots.append(dict(qkv=qkv, g=g, beta=beta, logits=lg, drafts=drafts, parent=parent))
    torch.cuda.synchronize(device)
    return slots


def run_gpu(args, w, world, rank, device):
    import torch
    from speculative_verify_gdn_gb300 import build as lib_build, inputs as I
    from speculative_verify_gdn_gb300.round import SpecRound

    lib_build.build()
    seed = rank_seed(args.seed, rank)
    cw = I.model_weights(w, seed, device)
    state, conv_state = I.initial_state(w, seed, device)
    pool = make_pool(w, seed, device, POOL)
    r = SpecRound(w, device)
    stream = torch.cuda.current_stream(device)
    fused = args.fused and not args.separate and w.accept != "tree"

    def step(k, rnd, evs=None):
        s = pool[k % POOL]
        if evs is not None:
            evs[0].record(stream)
        if fused:
            # the previous round's rollback and this round's verify, one pass over the state
            r.rollback_verify(s["qkv"], cw, conv_state, s["g"], s["beta"], state)
        else:
            r.verify(s["qkv"], cw, conv_state, s["g"], s["beta"], state, parent=s["parent"])
        if evs is not None:
            evs[1].record(stream)
        r.accept(s["logits"], s["drafts"], round_=rnd, seed=seed, parent=s["parent"])
        if evs is not None:
            evs[2].record(stream)
        if not fused:
            r.rollback(s["qkv"], s["g"], state, conv_state)
        if evs is not None:
            evs[3].record(stream)

    for k in range(args.warmup):
        step(k, k)
    r.check_status()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    # nlog[k]: accepted counts after timed step k; nlog0: after the last warm-up step (the counts
    # the first timed fused step commits)
    nlog0 = r.n_acc.clone()
    nlog = torch.zeros((K, w.B), dtype=torch.int32, device=device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device.index if device.index is not None else 0)
    clocks.start()
    barrier(device)
    torch.cuda.synchronize(device)
    start.record(stream)
    for k in range(K):
        step(args.warmup + k, args.warmup + k, evs[k])
        nlog[k].copy_(r.n_acc, non_blocking=True)
    end.record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    clk = clocks.stop()
    r.check_status()
    ms_total = start.elapsed_time(end)
    ms_total = reduce_max(ms_total, device)
    ms_step = ms_total / K
    t_ver = [evs[k][0].elapsed_time(evs[k][1]) for k in range(K)]
    t_acc = [evs[k][1].elapsed_time(evs[k][2]) for k in range(K)]
    t_rb = [evs[k][2].elapsed_time(evs[k][3]) for k in range(K)]
    nl = nlog.cpu().numpy()

    peak, peak_kind = read_peaks()
    ba = statistics.mean(bytes_accept(w, nl[k]) for k in range(K))
    if fused:
        nprev = [nlog0.cpu().numpy()] + [nl[k] for k in range(K - 1)]
        brv = [bytes_rollback_verify(w, nprev[k]) for k in range(K)]
        kern = {
            "gdn_rollback_verify": {"ms": statistics.mean(t_ver), "bytes": statistics.mean(brv)},
            "spec_accept": {"ms": statistics.mean(t_acc), "bytes": ba},
        }
        step_bytes = statistics.mean(brv) + ba
    else:
        bv = bytes_verify(w)
        brb = [bytes_rollback(w, nl[k]) for k in range(K)]
        kern = {
            "gdn_verify": {"ms": statistics.mean(t_ver), "bytes": bv},
            "spec_accept": {"ms": statistics.mean(t_acc), "bytes": ba},
            "gdn_rollback": {"ms": statistics.mean(t_rb), "bytes": statistics.mean(brb)},
        }
        step_bytes = bv + ba + statistics.mean(brb)
    # the accept's bytes are the rows its loop reaches; beside them, every row of the call (what
    # a pass over all N + 1 rows, such as the greedy kernels', reads)
    io = 2 if str(w.io_dtype).endswith("bfloat16") else 4
    kern["spec_accept"]["bytes_all_rows"] = w.B * (w.N + 1) * w.V * io + 4 * w.B * (2 * w.N + 2)
    for name, e in kern.items():
        e["GBps"] = e["bytes"] / (e["ms"] / 1e3) / 1e9
        e["frac_of_%s_peak" % peak_kind] = e["GBps"] / peak
        if "bytes_all_rows" in e:
            e["frac_all_rows"] = e["bytes_all_rows"] / (e["ms"] / 1e3) / 1e9 / peak
    dom = max(kern, key=lambda n: kern[n]["ms"])
    roof = {"bound": "hbm", "kernel": dom, "achieved": kern[dom]["GBps"], "peak": peak,
            "peak_source": "MEASURED_PEAKS.json hbm_gbs (%s)" % peak_kind, "unit": "GB/s",
            "frac": kern[dom]["GBps"] / peak,
            "traffic": profiled_traffic(w.name, dom) if full_size(args) else None,
            "algorithmic_bytes_per_launch": kern[dom]["bytes"],
            "step_frac": step_bytes / (ms_step / 1e3) / 1e9 / peak}
    mean_n = float(nl.mean())
    res = dict(ms_step=ms_step, kernels=kern, roofline=roof, clocks=clk, mean_n=mean_n,
               launches=K * r.launches_per_step(fused), ms_total=ms_total, fused=fused)

    # ---- the same steps launched from CUDA graphs
    if args.graph:
        res["graph"] = run_graph(args, w, r, pool, step, device)
        res["graph"]["gpu_launches"] = res["launches"]

    # ---- end to end: host (pinned) inputs copied in, results copied out, every step
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, w, r, pool, cw, state, conv_state, device, seed, fused)
    return res


def run_graph(args, w, r, pool, step, device):
    """The timed steps again, each launched as one CUDA graph replay instead of its calls one by
    one: one graph per input-pool slot, captured in the order the slots come after the steps run
    so far (so a fused step's double-buffered tape alternates as it does eagerly), each graph
    holding the step's kernels and a copy of its accepted counts. The round counter the sampling
    draws use is a launch argument, fixed at capture: the draws repeat every pool length, and the
    accepted counts are logged, as in the eager loop."""
    import torch
    stream = torch.cuda.current_stream(device)
    done = args.warmup + args.steps
    logs = [torch.empty_like(r.n_acc) for _ in range(POOL)]
    graphs = []
    torch.cuda.synchronize(device)
    for j in range(POOL):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(done + j, done + j)
            logs[j].copy_(r.n_acc)
        graphs.append(g)
    K = args.steps
    for j in range(max(args.warmup, POOL)):
        graphs[j % POOL].replay()
    r.check_status()
    nlog = torch.zeros((K, w.B), dtype=torch.int32, device=device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize(device)
    base = max(args.warmup, POOL)
    start.record(stream)
    for k in range(K):
        graphs[(base + k) % POOL].replay()
        nlog[k].copy_(logs[(base + k) % POOL], non_blocking=True)
    end.record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    r.check_status()
    ms = reduce_max(start.elapsed_time(end), device) / K
    world = dist_env()[0]
    return {"value": aggregate_tokens_per_s(world, w.B, w.N, ms), "unit": UNIT,
            "ms_per_step": ms, "steps": K, "graphs": POOL,
            "mean_accepted": float(nlog.float().mean().item())}


def run_e2e(args, w, r, pool, cw, state, conv_state, device, seed, fused=False):
    """The round through the public API with host-resident inputs, as a serving loop runs it:
    each step's inputs are copied from pinned host memory on a copy stream (step k+1's copy
    overlaps step k's kernels; three device sets, since a fused step also reads the previous
    round's set) and the accept results are copied back after each step. Every copy of the K
    steps lies inside the timed region."""
    import torch
    keys = ("qkv", "g", "beta", "logits", "drafts")
    host = []
    for s in pool[:2]:
        host.append({k: s[k].cpu().pin_memory() for k in keys})
    NS = 3
    devs = [{k: torch.empty_like(pool[0][k]) for k in keys} for _ in range(NS)]
    parent = pool[0]["parent"]
    out_h = torch.empty((w.B, r.out_tokens.shape[1]), dtype=torch.int32).pin_memory()
    n_h = torch.empty((w.B,), dtype=torch.int32).pin_memory()
    stream = torch.cuda.current_stream(device)
    # several copy streams, each taking a slice of every input (more than one copy engine)
    NCS = max(1, args.e2e_copy_streams)
    copy_streams = [torch.cuda.Stream(device) for _ in range(NCS)]
    copied = [[torch.cuda.Event() for _ in range(NCS)] for _ in range(NS)]
    done = [torch.cuda.Event() for _ in range(NS)]
    h2d = sum(host[0][k].numel() * host[0][k].element_size() for k in keys)
    d2h = out_h.numel() * 4 + n_h.numel() * 4
    K = max(3, min(args.steps, args.e2e_steps))

    def issue_copy(k):
        hs, dev = host[k % len(host)], devs[k % NS]
        for c, cs in enumerate(copy_streams):
            with torch.cuda.stream(cs):
                if k >= 2:
                    cs.wait_event(done[(k - 2) % NS])        # this set's last readers are done
                for key in keys:
                    n0 = hs[key].shape[0]
                    lo, hi = n0 * c // NCS, n0 * (c + 1) // NCS
                    if hi > lo:
                        dev[key][lo:hi].copy_(hs[key][lo:hi], non_blocking=True)
                copied[k % NS][c].record(cs)

    def run_step(k):
        dev = devs[k % NS]
        for ev in copied[k % NS]:
            stream.wait_event(ev)
        if fused:
            r.step_fused(dev["qkv"], dev["g"], dev["beta"], dev["logits"], dev["drafts"], cw,
                         state, conv_state, round_=k, seed=seed)
        else:
            r.step(dev["qkv"], dev["g"], dev["beta"], dev["logits"], dev["drafts"], cw, state,
                   conv_state, round_=k, seed=seed, parent=parent)
        done[k % NS].record(stream)
        n_h.copy_(r.n_acc, non_blocking=True)
        out_h.copy_(r.out_tokens, non_blocking=True)

    def run(nsteps, t0=None):
        if t0 is not None:
            for cs in copy_streams:
                cs.wait_event(t0)                          # the first copies start after t0
        issue_copy(0)
        for k in range(nsteps):
            if k + 1 < nsteps:
                issue_copy(k + 1)
            run_step(k)

    run(2)
    torch.cuda.synchronize(device)
    barrier(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    run(K, t0)
    t1.record(stream)
    torch.cuda.synchronize(device)
    ms = reduce_max(t0.elapsed_time(t1), device) / K
    world = dist_env()[0]
    return {"value": aggregate_tokens_per_s(world, w.B, w.N, ms), "unit": UNIT,
            "ms_per_step": ms, "steps": K, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": "inputs on %d copy streams, step k+1's overlapping step k's kernels" % NCS}


# ------------------------------------------------------------------------------ main
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fused", action="store_true",
                    help="time the fused step (gdn_rollback_verify + accept) instead of the "
                         "default three calls (verify / accept / rollback)")
    ap.add_argument("--separate", action="store_true",
                    help="the three calls (the default; overrides --fused)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--e2e-copy-streams", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (smaller profiling cases)")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the workload's layer count (smaller profiling cases)")
    ap.add_argument("--attn", default=None,
                    help="time the attention layers instead (an ATTN_WORKLOADS key, e.g. "
                         "qwen36_attn_b64_n8)")
    ap.add_argument("--hybrid", default=None,
                    help="time a whole hybrid round: the GDN workload plus this attention workload "
                         "(e.g. qwen36_attn_b64_n8)")
    ap.add_argument("--graph", action="store_true",
                    help="also time the steps launched as CUDA graph replays")
    ap.add_argument("--gate-dk", action="store_true",
                    help="one gate per key channel (g [L, B, T, Hv, d]); chain workloads only")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the bounded runs of the other single-GPU workloads that the default "
                         "run appends to its line (other_workloads)")
    ap.add_argument("--others-steps", type=int, default=200)
    args = ap.parse_args(argv)

    if args.attn:
        return run_attn(args)
    if args.hybrid:
        return run_hybrid(args)
    from speculative_verify_gdn_gb300 import inputs as I
    w = I.WORKLOADS[args.config]
    if args.batch is not None or args.layers is not None:
        w = I.custom(w, name=w.name, B=args.batch or w.B, L=args.layers or w.L)
    if args.gate_dk:
        if w.accept == "tree":
            raise SystemExit("--gate-dk: per-key-channel gates are built for chains")
        w = I.custom(w, name=w.name + "_gdk", gate_dk=True)
    ws, rank, local = dist_env()

    if args.impl == "reference":
        if ws > 1:
            init_dist("gloo")
            if rank != 0:
                return 0
        return run_reference(args, w)

    import torch
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    world, rank = init_dist("nccl")
    res = run_gpu(args, w, world, rank, device)
    cfg = workload_description(w)
    cfg["step"] = ("gdn_rollback_verify (the previous round's tape-replay rollback and this "
                   "round's verify, one pass over the state) + spec_accept" if res["fused"] else
                   "gdn_verify + spec_accept + gdn_rollback")
    line = {
        "metric": METRIC, "value": aggregate_tokens_per_s(world, w.B, w.N, res["ms_step"]),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": res["ms_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16", "data": "synthetic",
        "config": cfg, "roofline": res["roofline"],
        "kernels": res["kernels"], "mean_accepted": res["mean_n"],
        "committed_tokens_per_s": world * w.B * (res["mean_n"] + 1) / (res["ms_step"] / 1e3),
        "gpu_launches": res["launches"], "clocks": res["clocks"],
        "e2e": res.get("e2e"),
    }
    if "graph" in res:
        line["graph"] = res["graph"]
    default_run = (args.config == DEFAULT_CONFIG and not (args.fused or args.gate_dk or args.graph)
                   and args.batch is None and args.layers is None)
    if world == 1 and default_run and not args.no_others:
        line["other_workloads"] = other_workloads(args, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle single-threaded, then on every host core (one sequence per thread)
        t1u, t1a, u1, _ = oracle_unit_times(w, args.seed, args.cpu_budget / 2, w.L, 1)
        ncores = host_cores()
        tnu, tna, un, thr = oracle_unit_times(w, args.seed, args.cpu_budget / 2, w.L, ncores)
        line["cpu_baseline"] = {
            "value": cpu_tokens_per_s(w, tnu, tna), "unit": UNIT, "cores": thr, "nproc": ncores,
            "kind": "oracle",
            "sample": "%d (layer, sequence) units of verify+rollback and %d sequences' accepts of "
                      "this workload, %d sequences at a time on %d oracle threads (fp64, OpenMP "
                      "over independent sequences): %.2f ms per unit, %.2f ms per accept of "
                      "throughput; tokens/s = N / (L * unit + accept)"
                      % (un, thr, thr, thr, tnu * 1e3, tna * 1e3),
            "single_core": {"value": cpu_tokens_per_s(w, t1u, t1a), "cores": 1,
                            "sample": "%d units (%.1f ms each) and one sequence's accept (%.1f "
                                      "ms), one thread" % (u1, t1u * 1e3, t1a * 1e3)}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def other_workloads(args, device):
    """Bounded runs of the other single-GPU workloads (the N = 16 sampling workload, the 32-node
    trees, both attention workloads), each timed as its own bench line would be but with fewer
    steps and no e2e leg, so that one default run records them all."""
    import argparse as _ap
    from speculative_verify_gdn_gb300 import inputs as I
    out = {}

    def brief(d, kernels):
        return {"value": d["value"], "unit": d["unit"], "ms_per_step": d["ms_per_step"],
                "steps": d["steps"], "warmup": d["warmup"],
                "kernels": {k: {"ms": v["ms"], "frac_of_measured_peak": v.get("frac_of_measured_peak")}
                            for k, v in kernels.items()},
                "roofline": {k: d["roofline"].get(k) for k in ("kernel", "achieved", "frac",
                                                                "step_frac") if k in d["roofline"]},
                "clocks": d.get("clocks")}
    for c in (3, 4):
        a2 = _ap.Namespace(**vars(args))
        a2.config, a2.steps, a2.warmup, a2.no_e2e, a2.graph = c, args.others_steps, 5, True, False
        w = I.WORKLOADS[c]
        res = run_gpu(a2, w, 1, 0, device)
        d = {"value": aggregate_tokens_per_s(1, w.B, w.N, res["ms_step"]), "unit": UNIT,
             "ms_per_step": res["ms_step"], "steps": a2.steps, "warmup": a2.warmup,
             "roofline": res["roofline"], "clocks": res["clocks"]}
        out[w.name] = dict(brief(d, res["kernels"]), workload=workload_description(w)["workload"])
    for name in ("qwen36_attn_b64_n8", "qwen36_attn_b16_n16"):
        a2 = _ap.Namespace(**vars(args))
        a2.attn, a2.steps, a2.warmup, a2.batch, a2.layers = name, max(args.others_steps // 2, 10), 5, None, None
        d = attn_line(a2)
        kernels = {k: dict(v, frac_of_measured_peak=(v["GBps"] / d["roofline"]["peak"]) if "GBps" in v else None)
                   for k, v in d["kernels"].items()}
        out[name] = dict(brief(d, kernels), metric=d["metric"])
    return out


ATTN_METRIC = ("attention-layer verified draft tokens/sec (KV append + causal GQA attention + "
               "KV truncation); % HBM roofline")


def bytes_attn(w, n0):
    """Algorithmic bytes of one attn_verify call: the appended key / value rows read and written,
    every attended key and value read once ((n0 + T) rows per (layer, sequence, kv head)), q read
    and o written (bf16)."""
    rows_new = w.L * w.B * w.T * w.Hkv * w.D * 2
    kv = sum(2 * (int(n) + w.T) * w.D * 2 for n in n0) * w.L * w.Hkv
    qo = 2 * w.L * w.B * w.T * w.Hq * w.D * 2
    return 2 * 2 * rows_new + kv + qo


def run_attn(args):
    print(json.dumps(attn_line(args)), flush=True)
    return 0


def attn_line(args):
    """The hybrid's attention layers: one step = attn_verify (append + attention, all layers) and
    attn_truncate. The accepted counts are zero, so every step appends to and attends over the
    same committed rows (constant work per step)."""
    import torch
    from speculative_verify_gdn_gb300 import _lib, build as lib_build, inputs as I
    w = I.ATTN_WORKLOADS[args.attn]
    if args.batch is not None or args.layers is not None:
        import dataclasses
        w = dataclasses.replace(w, B=args.batch or w.B, L=args.layers or w.L)
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    lib_build.build()
    sh = _lib.AttnShape(L=w.L, B=w.B, T=w.T, Hq=w.Hq, Hkv=w.Hkv, D=w.D, ctx=w.ctx)
    kc, vc = I.attn_cache(w, args.seed, device)
    vt = _lib.vt_from_v(vc)
    del vc
    kv_len = I.attn_lengths(w).to(device)
    pool = [I.attn_round(w, k, args.seed, device) for k in range(POOL)]
    out = torch.empty(sh.q_shape(), dtype=torch.bfloat16, device=device)
    nws = _lib.attn_workspace_bytes(sh)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=device) if nws else None
    n_acc = torch.zeros(w.B, dtype=torch.int32, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)

    def step(k, evs=None):
        q, kn, vn = pool[k % POOL]
        if evs is not None:
            evs[0].record(stream)
        _lib.attn_verify(sh, q, kn, vn, kc, vt, kv_len, out, workspace=ws, status=status)
        if evs is not None:
            evs[1].record(stream)
        _lib.attn_truncate(n_acc, kv_len, w.T, status=status)
        if evs is not None:
            evs[2].record(stream)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize(device)
    assert int(status.item()) == 0, _lib.decode_status(int(status.item()))
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(0)
    clocks.start()
    torch.cuda.synchronize(device)
    start.record(stream)
    for k in range(K):
        step(args.warmup + k, evs[k])
    end.record(stream)
    torch.cuda.synchronize(device)
    clk = clocks.stop()
    assert int(status.item()) == 0, _lib.decode_status(int(status.item()))
    ms_step = start.elapsed_time(end) / K
    t_att = statistics.mean(evs[k][0].elapsed_time(evs[k][1]) for k in range(K))
    t_tr = statistics.mean(evs[k][1].elapsed_time(evs[k][2]) for k in range(K))
    peak, peak_kind = read_peaks()
    n0 = I.attn_lengths(w).tolist()
    ba = bytes_attn(w, n0)
    achieved = ba / (t_att / 1e3) / 1e9
    splits = 1 if not nws else None
    line = {
        "metric": ATTN_METRIC, "value": w.B * w.T / (ms_step / 1e3), "unit": UNIT, "n_gpus": 1,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s: %d attention layers (Qwen3.6-shaped: %d query heads over %d kv "
                               "heads of dim %d), batch %d, T=%d verify positions, %d committed "
                               "cache rows (capacity %d); accepted counts 0, so the work per step "
                               "is constant" % (w.name, w.L, w.Hq, w.Hkv, w.D, w.B, w.T,
                                                w.lengths[0], w.ctx),
                   "l2": "inputs larger than L2: %.2f GB of K / V cache read every step"
                         % (sum(2 * (n + w.T) * w.D * 2 for n in n0) * w.L * w.Hkv / 1e9),
                   "key_splits": "none" if splits == 1 else "flash-decoding split + combine"},
        "roofline": {"bound": "hbm", "kernel": "attn_verify", "achieved": achieved, "peak": peak,
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (%s)" % peak_kind, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": profiled_traffic(w.name, "attn_verify") if full_size(args) else None,
                     "algorithmic_bytes_per_launch": ba},
        "kernels": {"attn_verify": {"ms": t_att, "bytes": ba, "GBps": achieved},
                    "attn_truncate": {"ms": t_tr}},
        "gpu_launches": K * (3 if nws == 0 else 4), "clocks": clk,
    }
    return line


HYBRID_METRIC = ("hybrid-round verified draft tokens/sec (30 GDN + 10 attention layers: verify, "
                 "accept, rollback + KV truncation); % HBM roofline")


def run_hybrid(args):
    """A whole hybrid round of the layers this library covers: gdn_verify (30 GDN layers),
    attn_verify (10 attention layers), spec_accept, gdn_rollback and attn_truncate with the same
    accepted counts. The committed cache length is reset to the workload's at the start of each
    step (a 256-byte device copy), so every step attends over the same context."""
    import torch
    from speculative_verify_gdn_gb300 import _lib, build as lib_build, inputs as I
    from speculative_verify_gdn_gb300.round import SpecRound
    w = I.WORKLOADS[args.config]
    aw = I.ATTN_WORKLOADS[args.hybrid]
    assert (aw.B, aw.T) == (w.B, w.N) and w.accept != "tree", "attention workload must match"
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    lib_build.build()
    seed = args.seed
    cw = I.model_weights(w, seed, device)
    state, conv_state = I.initial_state(w, seed, device)
    pool = make_pool(w, seed, device, POOL)
    apool = [I.attn_round(aw, k, seed, device) for k in range(POOL)]
    kc, vc = I.attn_cache(aw, seed, device)
    vt = _lib.vt_from_v(vc)
    del vc
    kv_base = I.attn_lengths(aw).to(device)
    kv_len = kv_base.clone()
    ash = _lib.AttnShape(L=aw.L, B=aw.B, T=aw.T, Hq=aw.Hq, Hkv=aw.Hkv, D=aw.D, ctx=aw.ctx)
    aout = torch.empty(ash.q_shape(), dtype=torch.bfloat16, device=device)
    nws = _lib.attn_workspace_bytes(ash)
    aws = torch.empty(max(nws, 16), dtype=torch.uint8, device=device) if nws else None
    r = SpecRound(w, device)
    stream = torch.cuda.current_stream(device)
    names = ("gdn_verify", "attn_verify", "spec_accept", "gdn_rollback", "attn_truncate")

    def step(k, evs=None):
        s, (q, kn, vn) = pool[k % POOL], apool[k % POOL]
        kv_len.copy_(kv_base, non_blocking=True)
        rec = (lambda i: evs[i].record(stream)) if evs is not None else (lambda i: None)
        rec(0)
        r.verify(s["qkv"], cw, conv_state, s["g"], s["beta"], state)
        rec(1)
        _lib.attn_verify(ash, q, kn, vn, kc, vt, kv_len, aout, workspace=aws, status=r.status)
        rec(2)
        r.accept(s["logits"], s["drafts"], round_=k, seed=seed)
        rec(3)
        r.rollback(s["qkv"], s["g"], state, conv_state)
        rec(4)
        _lib.attn_truncate(r.n_acc, kv_len, aw.T, status=r.status)
        rec(5)

    for k in range(args.warmup):
        step(k)
    r.check_status()
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    nlog = torch.zeros((K, w.B), dtype=torch.int32, device=device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(0)
    clocks.start()
    torch.cuda.synchronize(device)
    start.record(stream)
    for k in range(K):
        step(args.warmup + k, evs[k])
        nlog[k].copy_(r.n_acc, non_blocking=True)
    end.record(stream)
    torch.cuda.synchronize(device)
    clk = clocks.stop()
    r.check_status()
    ms_step = start.elapsed_time(end) / K
    t = {n: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(K))
         for i, n in enumerate(names)}
    nl = nlog.cpu().numpy()
    peak, peak_kind = read_peaks()
    by = {"gdn_verify": bytes_verify(w), "attn_verify": bytes_attn(aw, kv_base.tolist()),
          "spec_accept": statistics.mean(bytes_accept(w, nl[k]) for k in range(K)),
          "gdn_rollback": statistics.mean(bytes_rollback(w, nl[k]) for k in range(K)),
          "attn_truncate": 8 * w.B}
    kern = {n: {"ms": t[n], "bytes": by[n], "GBps": by[n] / (t[n] / 1e3) / 1e9,
                "frac_of_%s_peak" % peak_kind: by[n] / (t[n] / 1e3) / 1e9 / peak} for n in names}
    dom = max(kern, key=lambda n: kern[n]["ms"])
    step_bytes = sum(by.values())
    line = {
        "metric": HYBRID_METRIC, "value": w.B * w.N / (ms_step / 1e3), "unit": UNIT, "n_gpus": 1,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "%s + %s: 30 GDN layers and 10 attention layers of the Qwen3.6 "
                               "hybrid, batch %d, N=%d, %d committed cache rows" % (
                                   w.name, aw.name, w.B, w.N, aw.lengths[0]),
                   "l2": "inputs larger than L2: %.2f GB moved per step" % (step_bytes / 1e9)},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": kern[dom]["GBps"], "peak": peak,
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (%s)" % peak_kind, "unit": "GB/s",
                     "frac": kern[dom]["GBps"] / peak,
                     "traffic": profiled_traffic(w.name if dom.startswith("gdn") else aw.name, dom),
                     "algorithmic_bytes_per_launch": by[dom],
                     "step_frac": step_bytes / (ms_step / 1e3) / 1e9 / peak},
        "kernels": kern, "mean_accepted": float(nl.mean()),
        "gpu_launches": K * (r.launches_per_step(False) + (2 if nws == 0 else 3) + 1),
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, w):
    """The oracle on the host cores, on this workload and metric; each step one (layer,
    sequence) unit of verify+rollback, plus one sequence's accept every L steps."""
    import numpy as np
    import oracle
    from speculative_verify_gdn_gb300 import inputs as I

    seed = args.seed
    # every host core: one sequence per oracle thread in each call
    nb = oracle.set_threads(host_cores())
    small = I.custom(w, name=w.name, L=1, B=nb)
    cw = I.model_weights(small, seed).double().numpy()
    st, cs = I.initial_state(small, seed)
    st, cs = st.double().numpy(), cs.double().numpy()
    d = oracle.OracleDims(L=1, B=nb, T=w.N, Hk=w.Hk, Hv=w.Hv, Dk=w.D, Dv=w.D, W=w.W)
    one = I.custom(w, name=w.name, B=nb)
    parent = tok = None
    if w.accept == "sample":
        lg, dr = I.sample_logits(one, 0, seed)
    elif w.accept == "tree":
        parent = I.random_tree(one, 0, seed).numpy()
        tok, lg, _ = I.tree_tokens_and_logits(one, I.random_tree(one, 0, seed), 0, seed)
        tok = tok.numpy()
    else:
        lg, dr, _ = I.greedy_logits(one, 0, seed)
    lgf = lg.float().numpy()
    streams = [I.round_stream(small, k, seed) for k in range(2)]
    streams = [tuple(t.double().numpy() for t in s) for s in streams]

    def step(k):
        qkv, g, beta = streams[k % 2]
        ref = oracle.verify(d, qkv, cw, cs, g, beta, st, parent=parent)
        path = None
        n = np.full(nb, max(1, w.N // 2), np.int32)
        if parent is not None:
            path = np.full((nb, w.P), -1, np.int32)
            path[:, 0] = 0
            n[:] = 1
        oracle.rollback(d, n, ref["tape_delta"], ref["tape_k"], g, qkv, st, cs, path=path)
        if k % w.L == w.L - 1:
            if w.accept == "sample":
                oracle.accept_sample(lgf, dr.numpy(), w.temperature, seed, k)
            elif w.accept == "tree":
                oracle.accept_tree(lgf, parent, tok, w.P)
            else:
                oracle.accept_greedy(lgf, dr.numpy())

    for k in range(args.warmup):
        step(k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        step(k)
    dt = time.perf_counter() - t0
    oracle.set_threads(1)
    ms_step = dt / args.steps * 1e3
    value = w.N * nb * (args.steps / w.L) / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_description(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle", "cores": nb,
                         "nproc": host_cores(),
                         "sample": "each step %d (layer, sequence) units of verify+rollback on %d "
                                   "oracle threads (one sequence each), %d sequences' accepts "
                                   "every %d steps; tokens/s = N x %d per %d steps"
                                   % (nb, nb, nb, w.L, nb, w.L)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
