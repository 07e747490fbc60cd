"""Benchmark of the batched verify-and-commit step on GB300.

Default workload: chain verification B=64, gamma=4 (5 target rows and 4
draft rows per request), V=128256, bf16 logits, temperature 0.8, top-k 50,
followed by the KV commit of every request's accepted prefix into a paged
bf16 cache (32 layers x 8 KV heads x 128, block 16, 2048-token prefix).  A
step is one spec_verify_chain + one spec_commit_kv over that batch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config {1..5}] [--impl ours|reference]

The metric is target rows verified per second, B*(gamma+1)/t (B*R/t for the
tree workload), with t the device time of one step; inputs are resident in
HBM when a step starts and L2 is flushed (a 256 MiB write) between steps.
`--impl reference` times the fp64 CPU oracle on this machine's cores on a
bounded sample of the same workload.  Under torchrun every rank runs its own
batch (weak scaling, no collective on the data path); the slowest rank's
time is used.

A single-GPU default run also times, each on its own workload and outside
the headline value, every other kernel with a bandwidth target (the greedy,
tree and full-vocabulary verify calls with their KV commits, the draft-tree
builder, the n-gram drafter) and reports them under "extra".
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from speculative_decoding_verification_37_gb300 import workloads as W  # noqa: E402

METRIC = "spec-verify rows/s + achieved HBM GB/s vs peak, B=64 γ=4 V=128256 bf16"
UNIT = "rows/s"
L2_FLUSH_BYTES = 256 << 20
CSRC = os.path.join(ROOT, "speculative_decoding_verification_37_gb300", "csrc")


def _code_only(src: str) -> str:
    """C/CUDA source with comments removed and whitespace collapsed, so that a
    comment edit does not invalidate a profile taken on the same code."""
    out, i, n = [], 0, len(src)
    while i < n:
        ch = src[i]
        if ch == '"' or ch == "'":  # literal: copy through its closing quote
            j = i + 1
            while j < n and src[j] != ch:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(ch)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (comments and layout ignored)."""
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, f), "r", encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_record(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, if it was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(f"{kernel} | {workload}")
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None
    return rec


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.path = None

    def start(self):
        import tempfile
        try:
            fd, self.path = tempfile.mkstemp(prefix=f"clocks_gpu{self.gpu}_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            text = f.read()
        os.unlink(self.path)  # the summary below goes into the JSON line
        for line in text.splitlines()[1:]:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1].split()[0]), float(parts[2].split()[0]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        smax = max(r[1] for r in rows)
        loaded = [r[0] for r in rows if r[0] > 0.5 * smax] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# workload setup on the device
# ---------------------------------------------------------------------------
class Workload:
    def __init__(self, cfg: int, seed: int, device, batch=None):
        import dataclasses
        self.cfg = cfg
        self.spec = W.WORKLOADS[cfg] if not batch else dataclasses.replace(W.WORKLOADS[cfg], B=batch)
        self.device = device
        s = self.spec
        if isinstance(s, W.TreeSpec):
            self.kind = "tree"
            tb = W.make_tree(s, seed=seed)
            self.host = tb
            self.rows = s.B * s.n_rows
            self.logit_bytes = s.logit_bytes()
            self.kvb = W.make_kv(s.kv, s.B, s.n_nodes + 1, seed=seed)
        else:
            self.kind = "chain"
            cb = W.make_chain(s, seed=seed)
            self.host = cb
            self.rows = s.B * (s.gamma + 1)
            self.logit_bytes = s.logit_bytes()
            self.kvb = W.make_kv(s.kv, s.B, s.gamma + 1, seed=seed) if s.kv else None
        self.B = s.B
        self._to_device()

    def _to_device(self):
        d = self.device
        h = self.host
        if self.kind == "tree":
            self.inputs = dict(logits=h.logits.to(d), node_token=torch.from_numpy(h.node_token).to(d),
                               node_parent=torch.from_numpy(h.node_parent).to(d),
                               row_of_node=torch.from_numpy(h.row_of_node).to(d))
        else:
            self.inputs = dict(target=h.target.to(d), draft_tokens=torch.from_numpy(h.draft_tokens).to(d))
            if h.draft is not None:
                self.inputs["draft"] = h.draft.to(d)
                self.inputs["uniforms"] = torch.from_numpy(h.uniforms).to(d)
        if self.kvb is not None:
            k = self.kvb
            self.inputs["temp_kv"] = k.temp_kv.to(d)
            self.inputs["block_table"] = torch.from_numpy(k.block_table).to(d)
            self.len0 = torch.from_numpy(k.committed_len.copy()).to(d)
            self.inputs["committed_len"] = self.len0.clone()
            self.cache = W.make_cache(k, device=d)

    def host_inputs(self):
        """Pinned host copies of every per-step input (for the end-to-end run)."""
        return {k: v.cpu().pin_memory() for k, v in self.inputs.items()}


def run_step(wl: Workload, inp, events=None, ws=None):
    """One verify (+ commit) step through the public API (allocates its
    outputs); used for the end-to-end measurement.  Returns the outputs."""
    from speculative_decoding_verification_37_gb300 import api
    s = wl.spec
    if wl.kind == "tree":
        out = api.verify_tree(inp["logits"], inp["node_token"], inp["node_parent"],
                              inp["row_of_node"], inp["committed_len"], R=s.n_rows)
        n_slots, slots = out.n_commit, out.commit_slots
    else:
        out = api.verify_chain(inp["target"], inp["draft_tokens"], gamma=s.gamma,
                               temperature=s.temperature, draft=inp.get("draft"),
                               uniforms=inp.get("uniforms"), top_k=s.top_k, accept_prob=False)
        n_slots, slots = out.n_out, None
    if wl.kvb is not None:
        api.commit_kv(inp["temp_kv"], wl.cache, inp["block_table"], n_slots, inp["committed_len"],
                      block_size=wl.kvb.kv.block_size, slots=slots)
    return out


class Step:
    """The timed step with every output and workspace preallocated, the
    verify call and the commit call each captured in a CUDA graph so that
    the timed region holds GPU work only (no allocation, no host latency).
    With ``in_place`` (chain only) the candidates' K/V are taken as written
    in place by the target forward: the verify call advances the lengths
    itself and there is no commit launch."""

    def __init__(self, wl: Workload, in_place: bool = False):
        from speculative_decoding_verification_37_gb300 import _lib as L
        from speculative_decoding_verification_37_gb300 import api
        self.wl = wl
        self.in_place = in_place
        s, dev, inp = wl.spec, wl.device, wl.inputs
        i32 = dict(dtype=torch.int32, device=dev)
        B = wl.B
        if wl.kind == "tree":
            if in_place:
                raise SystemExit("--kv-commit inplace applies to chain workloads (a tree's kept "
                                 "path is not a contiguous run of its candidates)")
            N, R = s.n_nodes, s.n_rows
            W_ = (N + 1 + 31) // 32
            self.out = dict(path=torch.empty((B, N), **i32), n_acc=torch.empty(B, **i32),
                            out_tokens=torch.empty((B, N + 1), **i32), n_out=torch.empty(B, **i32),
                            tree_mask=torch.empty((B, N + 1, W_), **i32),
                            pos=torch.empty((B, N + 1), **i32), commit_slots=torch.empty((B, N + 1), **i32),
                            n_commit=torch.empty(B, **i32), flags=torch.empty(B, **i32))
            self.ws = L.new_workspace(L.SPEC_WS_TREE, B, R, s.V, dev)

            def verify():
                L.spec_verify_tree(logits=inp["logits"], R=R, node_token=inp["node_token"],
                                   node_parent=inp["node_parent"], row_of_node=inp["row_of_node"],
                                   committed_len=inp["committed_len"], workspace=self.ws, **self.out)
            self.n_slots, self.slots = self.out["n_commit"], self.out["commit_slots"]
        else:
            g = s.gamma
            self.out = dict(n_acc=torch.empty(B, **i32), out_tokens=torch.empty((B, g + 1), **i32),
                            n_out=torch.empty(B, **i32), flags=torch.empty(B, **i32))
            kind = api.chain_workspace_kind(not s.greedy, s.top_k, s.V)
            self.ws = L.new_workspace(kind, B, g, s.V, dev)
            ip = {}
            if in_place:
                if wl.kvb is None:
                    raise SystemExit("--kv-commit inplace needs a workload with a KV cache")
                bs = wl.kvb.kv.block_size
                self.dlen0 = wl.len0 + g
                self.draft_len = self.dlen0.clone()
                ip = dict(committed_len=inp["committed_len"], draft_len=self.draft_len,
                          blocks_in_use=torch.empty(B, **i32), block_size=bs,
                          kv_capacity=wl.kvb.max_blocks * bs)

            def verify():
                L.spec_verify_chain(target_logits=inp["target"], draft_tokens=inp["draft_tokens"],
                                    workspace=self.ws, gamma=g, temperature=s.temperature,
                                    draft_logits=inp.get("draft"), uniforms=inp.get("uniforms"),
                                    top_k=s.top_k, **self.out, **ip)
            self.n_slots, self.slots = self.out["n_out"], None
        self.verify = verify
        self.commit = None
        if wl.kvb is not None and not in_place:
            self.cws = L.new_workspace(L.SPEC_WS_COMMIT, B, 0, 0, dev)

            def commit():
                L.spec_commit_kv(temp_kv=inp["temp_kv"], cache=wl.cache, block_table=inp["block_table"],
                                 n_slots=self.n_slots, committed_len=inp["committed_len"],
                                 block_size=wl.kvb.kv.block_size, workspace=self.cws, slots=self.slots)
            self.commit = commit
        self.graphs = None

    def reset(self):
        if self.wl.kvb is not None:
            self.wl.inputs["committed_len"].copy_(self.wl.len0)
        if self.in_place:
            self.draft_len.copy_(self.dlen0)

    def eager(self):
        self.reset()
        self.verify()
        if self.commit:
            self.commit()

    def capture(self):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(2):
                self.eager()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.gv = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.gv):
            self.verify()
        self.gc = None
        if self.commit:
            self.reset()
            self.gc = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.gc):
                self.commit()
        torch.cuda.synchronize()

    def replay(self, events=None):
        if events:
            events[0].record()
        self.gv.replay()
        if events:
            events[1].record()
        if self.gc is not None:
            self.gc.replay()
        if events:
            events[2].record()


def kv_bytes(wl: Workload, n_slots_total: int) -> int:
    return 0 if wl.kvb is None else 2 * wl.kvb.kv.token_bytes * n_slots_total


def kernel_name(wl: Workload) -> str:
    """The kernels one verify call of this workload launches."""
    from speculative_decoding_verification_37_gb300 import _lib as L
    if wl.kind == "tree" or wl.spec.greedy:
        return "argmax_pass_kernel+argmax_decide_kernel"
    if 0 < wl.spec.top_k <= L.TOPK_FAST_MAX:
        return "chain_topk_pass_kernel+chain_topk_decide_kernel"
    if (wl.spec.top_k == 0 or wl.spec.top_k >= wl.spec.V) and \
            wl.rows * -(-wl.spec.V * wl.spec.esize // 4096) >= 1024:
        return "chain_full_kernel"  # the persistent full-vocabulary path (at least 1,024 4 KiB items)
    return "chain_sample_kernel"


def time_steps(step: "Step", steps: int, warmup: int, flush):
    """Warm-up replays, then `steps` timed replays with the L2 flushed before
    each; returns the per-step (step, verify, commit) times in ms."""
    for _ in range(warmup):
        step.reset()
        step.replay()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        step.reset()
        flush.zero_()
        step.replay(events=ev[i])
    torch.cuda.synchronize()
    return ([e[0].elapsed_time(e[2]) for e in ev], [e[0].elapsed_time(e[1]) for e in ev],
            [e[1].elapsed_time(e[2]) for e in ev])


def verify_workload_record(cfg: int, dev, steps: int, warmup: int, flush, peak: float) -> dict:
    """Times workload `cfg`'s verify (+ commit) step on its own and returns
    the kernels' device times, algorithmic bytes and fractions of the peak."""
    wl = Workload(cfg, seed=0, device=dev)
    step = Step(wl)
    step.capture()
    step_ms, verify_ms, commit_ms = time_steps(step, steps, warmup, flush)
    t_v = statistics.mean(verify_ms)
    rec = {"workload": wl.spec.name, "kernel": kernel_name(wl), "verify_ms": round(t_v, 5),
           "algorithmic_bytes": wl.logit_bytes,
           "achieved_gbs": round(wl.logit_bytes / (t_v * 1e-3) / 1e9, 1),
           "frac": round(wl.logit_bytes / (t_v * 1e-3) / 1e9 / peak, 4),
           "rows_per_s": wl.rows / (statistics.mean(step_ms) * 1e-3), "steps": steps}
    if wl.kvb is not None:
        n_commit = int(step.n_slots.sum().item())
        t_c = statistics.mean(commit_ms)
        kvb = kv_bytes(wl, n_commit)
        rec.update(commit_kernel="commit_kv_kernel", commit_ms=round(t_c, 5), commit_bytes=kvb,
                   commit_frac=round(kvb / (t_c * 1e-3) / 1e9 / peak, 4), committed_tokens=n_commit)
    del step, wl
    torch.cuda.empty_cache()
    return rec


# ---------------------------------------------------------------------------
# CPU oracle (bounded sample)
# ---------------------------------------------------------------------------
def oracle_sample(cfg: int, seconds: float = 12.0, seed: int = 0, n_gen: int = 16,
                  wall_cap: float = 60.0, first: int = 0, start=None):
    """Times the fp64 oracle (verify + commit of each request) on this host,
    one request at a time: the inputs of `n_gen` requests of the workload
    (from request `first` on, wrapping around the batch) are generated once,
    then the oracle cycles over them until it has run for about `seconds` (or
    the wall clock reaches `wall_cap`).  `start` (a barrier) is waited on
    after the generation, so that parallel workers time the same interval.
    Returns (rows/s, sample text, requests run)."""
    import oracle as O
    spec = W.WORKLOADS[cfg]
    reqs = sorted({(first + i) % spec.B for i in range(min(spec.B, n_gen))})
    if isinstance(spec, W.TreeSpec):
        tb = W.make_tree(spec, seed=seed, requests=reqs)
        kvb = W.make_kv(spec.kv, len(reqs), spec.n_nodes + 1, seed=seed)
    else:
        tb = W.make_chain(spec, seed=seed, requests=reqs)
        kvb = W.make_kv(spec.kv, len(reqs), spec.gamma + 1, seed=seed) if spec.kv else None
    if kvb is not None:
        k = kvb.kv
        # the commit only reaches each request's tail blocks: a compact cache holds them
        tails = sorted(set(int(x) for x in kvb.block_table.reshape(-1)) - {0})
        remap = {blk: i + 1 for i, blk in enumerate(tails)}
        table = np.vectorize(lambda x: remap.get(int(x), 0))(kvb.block_table).astype(np.int32)
        cache0 = np.full((k.layers, 2, len(tails) + 1, k.block_size, k.heads, k.head_dim),
                         W.KV_SENTINEL, np.int16)
        temp = kvb.temp_kv.view(torch.int16).numpy()
    rows_done = n_req = passes = 0
    elapsed = 0.0
    if start is not None:
        start.wait()
    wall0 = time.perf_counter()
    while elapsed < seconds and time.perf_counter() - wall0 < wall_cap:
        cache = cache0.copy() if kvb is not None else None  # every pass commits into a fresh cache
        t0 = time.perf_counter()
        for i in range(len(reqs)):  # i indexes the generated (compacted) batch
            if isinstance(spec, W.TreeSpec):
                r = O.verify_tree(tb.logits_f64(i), tb.node_token[i], tb.node_parent[i],
                                  tb.row_of_node[i], int(kvb.committed_len[i]))
                slots = r.commit_slots
                rows_done += spec.n_rows
            elif spec.greedy:
                r = O.verify_chain_greedy(tb.target_f64(i), tb.draft_tokens[i])
                slots = O.chain_commit_slots(r.n_acc)
                rows_done += spec.gamma + 1
            else:
                r = O.verify_chain_sampled(tb.target_f64(i), tb.draft_f64(i), tb.draft_tokens[i],
                                           tb.uniforms[i].astype(np.float64), spec.temperature,
                                           spec.top_k)
                slots = O.chain_commit_slots(r.n_acc)
                rows_done += spec.gamma + 1
            if kvb is not None:
                O.commit_kv(cache, temp[i], table[i], slots, len(slots), int(kvb.committed_len[i]),
                            kvb.kv.block_size)
            n_req += 1
            if elapsed + (time.perf_counter() - t0) >= seconds:
                break
        elapsed += time.perf_counter() - t0
        passes += 1
    sample = (f"{n_req} request verifications + KV commits over {len(reqs)} requests of "
              f"this workload ({passes} passes), {elapsed:.1f} s of oracle time on one core "
              f"(input generation excluded)")
    return rows_done / elapsed, sample, n_req


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_worker(q, start, cfg, seconds, first, n_gen):
    try:
        v, _, n = oracle_sample(cfg, seconds=seconds, n_gen=n_gen, first=first, start=start)
        q.put((v, n, None))
    except BaseException as e:  # reported by the parent
        start.abort()
        q.put((0.0, 0, repr(e)))


def oracle_parallel(cfg: int, workers: int, seconds: float, n_gen: int = 4):
    """The oracle on `workers` processes at once (spawned, one thread each),
    each over its own requests of the workload, all timed over the same
    interval after their inputs are generated.  Returns (rows/s summed over
    the workers, sample text, requests run)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")  # never fork a process that may hold a CUDA context
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        q = ctx.Queue()
        start = ctx.Barrier(workers)
        procs = [ctx.Process(target=_oracle_worker, args=(q, start, cfg, seconds, w * n_gen, n_gen))
                 for w in range(workers)]
        for p in procs:
            p.start()
        res = [q.get(timeout=seconds + 600) for _ in procs]
        for p in procs:
            p.join(timeout=60)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    errs = [e for _, _, e in res if e]
    if errs:
        raise RuntimeError(f"oracle worker failed: {errs[0]}")
    total = sum(v for v, _, _ in res)
    n_req = sum(n for _, n, _ in res)
    sample = (f"{n_req} request verifications + KV commits on {workers} processes at once (one thread "
              f"each, {n_gen} requests of this workload per process), about {seconds:.0f} s each, "
              f"rows/s summed over the processes (input generation excluded)")
    return total, sample, n_req


def cpu_baseline_record(cfg: int, seconds: float = 10.0):
    """The oracle timed on this host's cores: single-threaded, then one
    process per core.  `value` and `cores` are the all-cores run's."""
    cores = host_cores()
    v1, s1, _ = oracle_sample(cfg, seconds=seconds)
    if cores > 1:
        vn, sn, _ = oracle_parallel(cfg, cores, seconds)
    else:
        vn, sn = v1, s1
    return {"value": vn, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sn,
            "host_cores": os.cpu_count(), "single_core": {"value": v1, "cores": 1, "sample": s1}}


# ---------------------------------------------------------------------------
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    dist.init_process_group(backend)
    return rank, ws, local


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def config_dict(cfg: int, world: int, batch: int = 0):
    import dataclasses
    s = W.WORKLOADS[cfg] if not batch else dataclasses.replace(W.WORKLOADS[cfg], B=batch)
    d = {"workload": s.name, "B_per_gpu": s.B, "V": s.V, "dtype": s.dtype,
         "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)",
         "parallelism": f"dp{world} (independent request shards, no collective)"}
    if isinstance(s, W.ChainSpec):
        d.update(gamma=s.gamma, temperature=s.temperature, top_k=s.top_k)
    else:
        d.update(topKSpec=[list(x) for x in s.topKSpec], topHead=list(s.topHead), rows=s.n_rows)
    if s.kv:
        d.update(kv=f"{s.kv.layers}L x {s.kv.heads}H x {s.kv.head_dim} bf16, block "
                    f"{s.kv.block_size}, prefix {s.kv.prefix}")
    return d


def run_reference(args, rank, world):
    if rank != 0:
        return
    cores = host_cores()
    seconds = min(60.0, max(2.0, 4.0 * args.steps))
    if cores > 1:
        v, sample, _ = oracle_parallel(args.config, cores, seconds)
    else:
        v, sample, _ = oracle_sample(args.config, seconds=seconds)
    s = W.WORKLOADS[args.config]
    dtype = s.dtype
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic", "config": config_dict(args.config, world),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


NGRAM_METRIC = "n-gram drafts: requests/s + history GB/s vs peak"


def ngram_times(run, d_hist, d_lens, steps, warmup, flush):
    """Device times (ms) of `steps` drafter launches, L2 flushed before each."""
    for _ in range(max(3, warmup)):
        run(d_hist, d_lens)
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run(d_hist, d_lens)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return times


def ngram_record(dev, steps, warmup, flush, peak) -> dict:
    """The drafter on its workload, timed on its own (for the default line)."""
    from speculative_decoding_verification_37_gb300 import api
    spec = W.NGRAM_SPEC
    hist, lens = W.make_histories(spec, seed=0)
    hist_bytes = int(lens.astype(np.int64).sum()) * 4
    d_hist, d_lens = torch.from_numpy(hist).to(dev), torch.from_numpy(lens).to(dev)
    run = lambda h, l: api.ngram_draft(h, l, gamma=spec.gamma, n_min=spec.n_min, n_max=spec.n_max)
    t = statistics.mean(ngram_times(run, d_hist, d_lens, steps, warmup, flush))
    del d_hist, d_lens
    torch.cuda.empty_cache()
    return {"workload": spec.name, "kernel": "ngram_draft_kernel", "ms": round(t, 5),
            "algorithmic_bytes": hist_bytes, "achieved_gbs": round(hist_bytes / (t * 1e-3) / 1e9, 1),
            "frac": round(hist_bytes / (t * 1e-3) / 1e9 / peak, 4),
            "requests_per_s": spec.B / (t * 1e-3), "steps": steps}


def run_ngram(args, rank, world, local):
    """The prompt-lookup drafter on a batch of long histories (one launch per
    step, histories resident; L2 flushed between steps)."""
    spec = W.NGRAM_SPEC
    hist, lens = W.make_histories(spec, seed=rank)
    hist_bytes = int(lens.astype(np.int64).sum()) * 4
    cfg = {"workload": spec.name, "B_per_gpu": spec.B, "max_len": spec.max_len, "V": spec.vocab,
           "gamma": spec.gamma, "n_min": spec.n_min, "n_max": spec.n_max,
           "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)",
           "parallelism": f"dp{world} (independent request shards, no collective)"}
    if args.impl == "reference":
        if rank == 0:
            v, sample = ngram_oracle_sample(hist, lens, spec, seconds=max(2.0, 2.0 * args.steps))
            print(json.dumps({"impl": "reference", "metric": NGRAM_METRIC, "value": v, "unit": "requests/s",
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
                              "data": "synthetic", "config": cfg,
                              "cpu_baseline": {"value": v, "unit": "requests/s", "cores": 1, "kind": "oracle",
                                               "sample": sample},
                              "e2e": {"value": v, "unit": "requests/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
        return
    from speculative_decoding_verification_37_gb300 import build as _b
    from speculative_decoding_verification_37_gb300 import api
    _b.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    d_hist = torch.from_numpy(hist).to(dev)
    d_lens = torch.from_numpy(lens).to(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    run = lambda h, l: api.ngram_draft(h, l, gamma=spec.gamma, n_min=spec.n_min, n_max=spec.n_max)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    barrier(world)
    times = ngram_times(run, d_hist, d_lens, args.steps, args.warmup, flush)
    barrier(world)
    clk = clocks.stop()
    t = max_over_ranks(statistics.mean(times), world)
    peak, peak_kind = measured_peaks()
    achieved = hist_bytes / (t * 1e-3) / 1e9
    e2e = None
    if not args.no_e2e:
        h_hist, h_lens = torch.from_numpy(hist).pin_memory(), torch.from_numpy(lens).pin_memory()
        et = []
        for i in range(5):
            flush.zero_()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            d_hist.copy_(h_hist, non_blocking=True)
            d_lens.copy_(h_lens, non_blocking=True)
            o = run(d_hist, d_lens)
            host = [o.draft_tokens.to("cpu", non_blocking=True), o.n_draft.to("cpu", non_blocking=True)]
            e1.record()
            torch.cuda.synchronize()
            if i >= 2:
                et.append(e0.elapsed_time(e1))
        te = max_over_ranks(statistics.mean(et), world)
        e2e = {"value": spec.B * world / (te * 1e-3), "unit": "requests/s",
               "h2d_bytes_per_step": hist.nbytes + lens.nbytes,
               "d2h_bytes_per_step": sum(h.numel() * h.element_size() for h in host),
               "ms_per_step": round(te, 4)}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, sample = ngram_oracle_sample(hist, lens, spec, seconds=8.0)
        cpu = {"value": v, "unit": "requests/s", "cores": 1, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps({"metric": NGRAM_METRIC, "value": spec.B * world / (t * 1e-3), "unit": "requests/s",
                          "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t, 5),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
                          "data": "synthetic", "config": cfg,
                          "roofline": {"bound": "hbm", "kernel": "ngram_draft_kernel", "achieved": round(achieved, 1),
                                       "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                                       "traffic": None, "algorithmic_bytes": hist_bytes,
                                       "avg_launch_ms": round(t, 5),
                                       "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)"},
                          "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps, "clocks": clk,
                          "kernel_source": kernel_source_hash()}), flush=True)


TREE_BUILD_METRIC = "draft trees built level by level: trees/s + draft-logit GB/s vs peak"


def tree_build_oracle_sample(levels, spec, seconds: float):
    """Times the oracle's tree build on this host, one request at a time over
    the batch's first requests, for about `seconds`."""
    import oracle as O
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < seconds and n < spec.B:
        rows = [lv[n * h:(n + 1) * h].double().numpy() for lv, h in zip(levels, spec.topHead)]
        O.build_tree(rows, spec.topKSpec, spec.topHead)
        n += 1
    el = time.perf_counter() - t0
    return n / el, (f"{n} trees of the batch ({spec.n_rows} draft rows of {spec.V} logits each), "
                    f"{el:.1f} s on one core")


def tree_build_graph(spec, d_levels, dev, warmup):
    """A TreeBuilder over the levels' draft rows, its three level calls
    captured in one CUDA graph and warmed up."""
    from speculative_decoding_verification_37_gb300 import api
    tb = api.TreeBuilder(spec.B, spec.V, spec.topKSpec, spec.topHead, dev)

    def build_all():
        for i, lv in enumerate(d_levels):
            tb.level(lv, i)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            build_all()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        build_all()
    for _ in range(max(3, warmup)):
        graph.replay()
    torch.cuda.synchronize()
    return tb, build_all, graph


def graph_times(graph, steps, flush):
    """Device times (ms) of `steps` replays, L2 flushed before each."""
    times = []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return times


def tree_build_record(dev, steps, warmup, flush, peak) -> dict:
    """The draft-tree builder on the tree workload's shape, timed on its own
    (for the default line)."""
    spec = W.WORKLOADS[4]
    levels = W.make_tree_levels(spec, seed=0)
    logit_bytes = sum(lv.numel() * lv.element_size() for lv in levels)
    d_levels = [lv.to(dev) for lv in levels]
    tb, _, graph = tree_build_graph(spec, d_levels, dev, warmup)
    t = statistics.mean(graph_times(graph, steps, flush))
    del graph, tb, d_levels
    torch.cuda.empty_cache()
    return {"workload": f"tree build {[list(k) for k in spec.topKSpec]}/{list(spec.topHead)} B={spec.B} "
                        f"V={spec.V} {spec.dtype}",
            "kernel": "tree_level_kernel+tree_merge_kernel (3 levels)", "ms": round(t, 5),
            "algorithmic_bytes": logit_bytes, "achieved_gbs": round(logit_bytes / (t * 1e-3) / 1e9, 1),
            "frac": round(logit_bytes / (t * 1e-3) / 1e9 / peak, 4), "trees_per_s": spec.B / (t * 1e-3),
            "steps": steps}


def run_tree_build(args, rank, world, local):
    """The draft-tree builder over the tree workload's shape: one step is the
    three level calls of a whole tree (captured in one CUDA graph), the draft
    rows resident; L2 flushed between steps."""
    import dataclasses
    spec = W.WORKLOADS[4] if not args.batch else dataclasses.replace(W.WORKLOADS[4], B=args.batch)
    levels = W.make_tree_levels(spec, seed=rank)
    logit_bytes = sum(lv.numel() * lv.element_size() for lv in levels)
    cfg = {"workload": f"tree build {[list(k) for k in spec.topKSpec]}/{list(spec.topHead)} "
                       f"B={spec.B} V={spec.V} {spec.dtype}",
           "B_per_gpu": spec.B, "V": spec.V, "dtype": spec.dtype,
           "topKSpec": [list(k) for k in spec.topKSpec], "topHead": list(spec.topHead),
           "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)",
           "parallelism": f"dp{world} (independent request shards, no collective)"}
    if args.impl == "reference":
        if rank == 0:
            v, sample = tree_build_oracle_sample(levels, spec, seconds=max(2.0, 2.0 * args.steps))
            print(json.dumps({"impl": "reference", "metric": TREE_BUILD_METRIC, "value": v, "unit": "trees/s",
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                              "dtype": spec.dtype, "data": "synthetic", "config": cfg,
                              "cpu_baseline": {"value": v, "unit": "trees/s", "cores": 1, "kind": "oracle",
                                               "sample": sample},
                              "e2e": {"value": v, "unit": "trees/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
        return
    from speculative_decoding_verification_37_gb300 import build as _b
    from speculative_decoding_verification_37_gb300 import api
    _b.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    d_levels = [lv.to(dev) for lv in levels]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    tb, build_all, graph = tree_build_graph(spec, d_levels, dev, args.warmup)
    # per-level launch times (eager, events between the calls)
    lvl_ms = [[] for _ in d_levels]
    for _ in range(3):
        flush.zero_()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(d_levels) + 1)]
        ev[0].record()
        for i, lv in enumerate(d_levels):
            tb.level(lv, i)
            ev[i + 1].record()
        torch.cuda.synchronize()
        for i in range(len(d_levels)):
            lvl_ms[i].append(ev[i].elapsed_time(ev[i + 1]))
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    barrier(world)
    times = graph_times(graph, args.steps, flush)
    barrier(world)
    clk = clocks.stop()
    t = max_over_ranks(statistics.mean(times), world)
    peak, peak_kind = measured_peaks()
    achieved = logit_bytes / (t * 1e-3) / 1e9
    # DRAM bytes of one whole build (all levels), from the committed capture
    tr = traffic_record("tree_level_kernel+tree_merge_kernel", cfg["workload"])
    e2e = None
    if not args.no_e2e:
        h_levels = [lv.pin_memory() for lv in levels]
        et = []
        for i in range(5):
            flush.zero_()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for d, h in zip(d_levels, h_levels):
                d.copy_(h, non_blocking=True)
            build_all()
            host = [x.to("cpu", non_blocking=True) for x in (tb.node_token, tb.node_parent, tb.row_of_node)]
            e1.record()
            torch.cuda.synchronize()
            if i >= 2:
                et.append(e0.elapsed_time(e1))
        te = max_over_ranks(statistics.mean(et), world)
        e2e = {"value": spec.B * world / (te * 1e-3), "unit": "trees/s", "h2d_bytes_per_step": logit_bytes,
               "d2h_bytes_per_step": sum(h.numel() * h.element_size() for h in host),
               "ms_per_step": round(te, 4)}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, sample = tree_build_oracle_sample(levels, spec, seconds=8.0)
        cpu = {"value": v, "unit": "trees/s", "cores": 1, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps({"metric": TREE_BUILD_METRIC, "value": spec.B * world / (t * 1e-3), "unit": "trees/s",
                          "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t, 5),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
                          "data": "synthetic", "config": cfg,
                          "roofline": {"bound": "hbm", "kernel": "tree_level_kernel+tree_merge_kernel",
                                       "achieved": round(achieved, 1),
                                       "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                                       "traffic": None if tr is None else tr["bytes_per_launch"],
                                       "algorithmic_bytes": logit_bytes,
                                       "avg_launch_ms": round(t / len(d_levels), 5),
                                       "unit_of_traffic_and_time": "one whole tree build (every level's "
                                                                   "pass and merge)",
                                       "level_ms": [round(statistics.mean(x), 5) for x in lvl_ms],
                                       "level_bytes": [lv.numel() * lv.element_size() for lv in levels],
                                       "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)"},
                          "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps * 2 * len(d_levels),
                          "clocks": clk, "kernel_source": kernel_source_hash()}), flush=True)


def ngram_oracle_sample(hist, lens, spec, seconds: float):
    """Times the oracle on this host, one request at a time over the batch's
    first requests, for about `seconds`."""
    import oracle as O
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < seconds and n < spec.B:
        O.ngram_draft(hist[n, :lens[n]].tolist(), spec.n_min, spec.n_max, spec.gamma)
        n += 1
    el = time.perf_counter() - t0
    return n / el, f"{n} requests of the batch (histories of up to {spec.max_len} tokens), {el:.1f} s on one core"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's request count (smaller cases for profiling)")
    ap.add_argument("--workload", default="verify", choices=["verify", "ngram", "tree_build"],
                    help="ngram: the prompt-lookup drafter on long token histories; tree_build: "
                         "the draft-tree builder on the tree workload's shape")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads' kernel lines (workloads 3-5, the tree builder, "
                         "the n-gram drafter) that a single-GPU default run adds under 'extra'")
    ap.add_argument("--kv-commit", default="copy", choices=["copy", "inplace"],
                    help="inplace (chain): K/V written in place by the forward, the verify "
                         "call advances the lengths, no commit kernel")
    args = ap.parse_args()
    rank, world, local = dist_setup()
    if args.workload == "ngram":
        run_ngram(args, rank, world, local)
        return
    if args.workload == "tree_build":
        run_tree_build(args, rank, world, local)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.warmup < 3:
        args.warmup = 3

    from speculative_decoding_verification_37_gb300 import build as _b
    from speculative_decoding_verification_37_gb300 import _lib as L
    _b.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = Workload(args.config, seed=rank, device=dev, batch=args.batch)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    in_place = args.kv_commit == "inplace"
    step = Step(wl, in_place=in_place)
    step.capture()

    # warm-up
    for _ in range(args.warmup):
        step.reset()
        step.replay()
    torch.cuda.synchronize()

    # timed steps: per-step events around the graph replays; the length reset
    # and the L2 flush (which also keeps the GPU busy while the host enqueues)
    # sit between the events
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    step_ms, verify_ms, commit_ms = time_steps(step, args.steps, 0, flush)
    barrier(world)
    clk = clocks.stop()
    n_commit_total = int(step.n_slots.sum().item()) if wl.kvb is not None else 0
    t_step = statistics.mean(step_ms)
    t_step_max = max_over_ranks(t_step, world)
    rows_total = wl.rows * world
    value = rows_total / (t_step_max * 1e-3)

    peak, peak_kind = measured_peaks()
    t_verify = statistics.mean(verify_ms)
    achieved = wl.logit_bytes / (t_verify * 1e-3) / 1e9
    kname = kernel_name(wl)
    tr = traffic_record(kname, config_dict(args.config, world, args.batch)["workload"])
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": None if tr is None else tr["bytes_per_launch"],
                "algorithmic_bytes": wl.logit_bytes, "avg_launch_ms": round(t_verify, 5),
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                else "fallback 6.8 TB/s"}
    commit = None
    if in_place:
        commit = {"kernel": None, "mode": "in place: the verify call advances committed_len, "
                  "draft_len and blocks_in_use; no K/V copy, no commit launch",
                  "committed_tokens": n_commit_total}
    elif wl.kvb is not None:
        t_commit = statistics.mean(commit_ms)
        kvb = kv_bytes(wl, n_commit_total)
        ctr = traffic_record("commit_kv_kernel", config_dict(args.config, world, args.batch)["workload"])
        commit = {"kernel": "commit_kv_kernel", "avg_launch_ms": round(t_commit, 5),
                  "algorithmic_bytes": kvb, "achieved_gbs": round(kvb / (t_commit * 1e-3) / 1e9, 1),
                  "frac": round(kvb / (t_commit * 1e-3) / 1e9 / peak, 4),
                  "traffic": None if ctr is None else ctr["bytes_per_launch"],
                  "committed_tokens": n_commit_total}

    # end-to-end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        hin = wl.host_inputs()
        h2d = sum(v.numel() * v.element_size() for v in hin.values())
        d_in = {k: torch.empty_like(v, device=dev) for k, v in hin.items()}
        e_steps = max(3, min(args.steps, 10))
        times = []
        d2h = 0
        for i in range(e_steps + 2):
            flush.zero_()
            torch.cuda.synchronize()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            for k, v in hin.items():
                d_in[k].copy_(v, non_blocking=True)
            o = run_step(wl, d_in)
            res = [o.n_acc, o.out_tokens, o.n_out] + ([d_in["committed_len"]] if wl.kvb else [])
            host = [r.to("cpu", non_blocking=True) for r in res]
            t1.record()
            torch.cuda.synchronize()
            d2h = sum(r.numel() * r.element_size() for r in host)
            if i >= 2:
                times.append(t0.elapsed_time(t1))
        t_e2e = max_over_ranks(statistics.mean(times), world)
        e2e = {"value": rows_total / (t_e2e * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(t_e2e, 4),
               "path": "pinned host -> device copies, spec_verify + spec_commit_kv, device -> host "
                       "of n_acc/out_tokens/n_out/committed_len, all in the timed region"}

    # every other kernel with a bandwidth target, each timed on its own
    # workload (single-GPU default runs only; not part of the headline value)
    extra = None
    if world == 1 and not args.no_extra and args.config == 2 and not args.batch and not in_place:
        x_steps = max(3, min(args.steps, 10))
        extra = {"note": "each kernel timed alone on its own workload (CUDA graphs, L2 flushed before "
                         f"each of {x_steps} steps); not part of the headline value",
                 "workloads": [verify_workload_record(c, dev, x_steps, 3, flush, peak) for c in (3, 4, 5)]}
        extra["workloads"].append(tree_build_record(dev, x_steps, 3, flush, peak))
        extra["workloads"].append(ngram_record(dev, x_steps, 3, flush, peak))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_record(args.config)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step_max, 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": W.WORKLOADS[args.config].dtype, "data": "synthetic",
                "config": config_dict(args.config, world, args.batch),
                "rounds_per_s": wl.B * world / (t_step_max * 1e-3),
                "step_gbs": round((wl.logit_bytes + kv_bytes(wl, n_commit_total)) /
                                  (t_step_max * 1e-3) / 1e9, 1),
                "roofline": roofline, "commit": commit, "cpu_baseline": cpu, "e2e": e2e, "extra": extra,
                "gpu_launches": args.steps * ((2 if "+" in kname else 1) +
                                              (1 if wl.kvb is not None and not in_place else 0)),
                "clocks": clk, "kernel_source": kernel_source_hash()}
        if in_place:
            line["config"]["kv_commit"] = "in place (length advance inside the verify call)"
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
