"""Throughput of the page-major KV pool's hot path on one GB300 (or N replicas).

One step is one pass of the whole path on the Llama-3-8B-shaped decode
workload (L=32 layers, 8 KV heads, head_dim 128, bf16, page size 16, 4096
pages = an 8 GiB pool):
  1. kv_translate          512 slots -> ids (256 decode tokens + 256 chunk tokens)
  2. kv_store_all_layers   the 256-token chunk into all 32 layers (one launch)
  3. kv_gather_plan        order the block table's entries by page (once per step)
  4. for each of the 32 layers:
       kv_store_layer      the 256 decode tokens (one per sequence)
       kv_gather_layer_planned  256 sequences x 4096 context tokens through the block tables
  5. kv_move               8192 tokens (all 64 row-blocks each) to new slots
Metric: useful GB/s = algorithmic bytes moved per step (every payload row read
once and written once, plus index bytes) / step time, with inputs resident in
HBM. The working set (8 GiB pool, 4 GiB of gather output per layer) is far
larger than L2, so no flush is needed between steps.

`--impl reference` times the CPU oracle (oracle/, plain C loops) on a bounded
sample of the same step on the host cores, same metric and unit.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

GB = 1e9
SHAPE = synth.SHAPES[2]
N_DECODE = 256          # sequences, one new token each
CTX = 4096              # context tokens per sequence
N_CHUNK = 256           # tokens of a prefill chunk stored into all layers at once
N_MOVE = 8192           # tokens moved per step
WORKLOAD = ("llama3-8b-decode: L=32 H_kv=8 D=128 bf16 ps=16 P=4096 (8 GiB pool); step = translate 512 slots, "
            "store_all_layers 256 chunk tokens, gather plan (page-major order of the block table), 32 x "
            "(store_layer 256 decode tokens + gather 256 seqs x 4096 tokens), move 8192 tokens x 64 row-blocks")


def gather_bytes(g: synth.GatherBatch, ps: int, R: int, kv_rows: int = 2) -> dict:
    """Bytes one gather launch of batch g moves, two ways.

    method: what the gather must move at the least -- every distinct source
    row the table names inside the windows read once (K and V), every output
    row written once, plus the table entries that cover the windows and the
    per-sequence start, length and output offset. This is the figure the HBM
    roofline bounds.
    per_reader: every output row's source counted once per reader (2R read +
    2R written per output token, plus 4/ps of table): a page that many
    sequences share is counted once per sequence, so this rate can exceed
    the HBM peak when L2 serves the repeats."""
    bt = np.asarray(g.block_table)
    st = np.asarray(g.seq_start, np.int64)
    ln = np.asarray(g.seq_len, np.int64)
    cnt = np.maximum(ln - st, 0)
    rows = int(cnt.sum())
    seq = np.repeat(np.arange(bt.shape[0]), cnt)
    j = np.arange(rows, dtype=np.int64) - np.repeat(np.cumsum(cnt) - cnt, cnt) + np.repeat(st, cnt)
    page = bt[seq, j // ps].astype(np.int64)
    tok = np.where(page < 0, -1, page * ps + j % ps)  # a tombstoned entry reads the one sink row
    distinct = int(np.unique(tok).size) if rows else 0
    first = st // ps
    last = np.where(cnt > 0, -(-ln // ps), first)
    entries = int(np.maximum(last - first, 0).sum())
    method = distinct * kv_rows * R + rows * kv_rows * R + entries * 4 + bt.shape[0] * (4 + 4 + 8)
    per_reader = rows * 2 * kv_rows * R + rows * 4 // ps
    return {"method": method, "per_reader": per_reader, "rows": rows, "distinct_source_rows": distinct,
            "table_entries": entries}


def step_bytes(g: synth.GatherBatch, shape=SHAPE, n_decode=N_DECODE, n_chunk=N_CHUNK, n_move=N_MOVE):
    """Method bytes of one step, by kernel (every row read once and written
    once, plus the index bytes each kernel must read), and the per-launch
    gather accounting (gather_bytes)."""
    L, R, ps = shape.layer_num, shape.row_bytes, shape.page_size
    gb = gather_bytes(g, ps, R)
    by_kernel = {
        "translate": (n_decode + n_chunk) * (8 + 4),
        "store_all_layers": n_chunk * (2 * L * R * 2 + 4),
        "store_layer": L * n_decode * (2 * R * 2 + 4),
        "gather": L * gb["method"],
        "move": n_move * (2 * L * R * 2 + 8),
    }
    return by_kernel, gb


# ------------------------------------------------------------------ inputs

def make_inputs(rank: int, shape=SHAPE, n_decode=N_DECODE, ctx=CTX, n_chunk=N_CHUNK, n_move=N_MOVE):
    """Seeded host inputs of one step (numpy)."""
    ps, P = shape.page_size, shape.num_pages
    rng = synth.rng_for(shape.seed + 7919 * rank, synth.S_MISC, 0)
    slots = synth.distinct_slots(rng, ps, P * ps, n_decode + n_chunk + 2 * n_move)
    dec, chunk = slots[:n_decode], slots[n_decode:n_decode + n_chunk]
    mv = slots[n_decode + n_chunk:]
    npg = ctx // ps
    bt = np.stack([1 + rng.permutation(P - 1)[:npg] for _ in range(n_decode)]).astype(np.int32)
    g = synth.GatherBatch(bt, np.zeros(n_decode, np.int32), np.full(n_decode, ctx, np.int32))
    kd, vd = synth.kv_pair(shape, shape.layer_num * n_decode, 0, seed=shape.seed + rank)
    kc, vc = synth.kv_pair(shape, shape.layer_num * n_chunk, 1, seed=shape.seed + rank)
    L, R = shape.layer_num, shape.row_bytes

    def rows(a, n):
        return np.ascontiguousarray(a).view(np.uint8).reshape(L, n, R)

    return dict(slots=np.concatenate([dec, chunk]).astype(np.int64), g=g,
                k_dec=rows(kd, n_decode), v_dec=rows(vd, n_decode),
                k_chunk=rows(kc, n_chunk), v_chunk=rows(vc, n_chunk),
                move_src=mv[:n_move], move_dst=mv[n_move:])


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str | None):
        self.proc = None
        self.lines: list[str] = []
        self.device_id = device_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.device_id:
            cmd += ["-i", self.device_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ peaks / profile

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


GATHER_SOURCES = [os.path.join(ROOT, "gather_translate_kv_gb300", "csrc", f)
                  for f in ("kv_gather.cu", "kv_common.cuh", "kv_plan.cuh", "kv_bulk.cuh")]
TRAFFIC_PROFILE = "gather_planned_decode_small_dram.txt"


def sources_hash(paths) -> str:
    """Short hash of the sources a kernel is built from."""
    import hashlib

    h = hashlib.sha256()
    for path in paths:
        h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(out_rows: int, summary=TRAFFIC_PROFILE, sources=GATHER_SOURCES):
    """DRAM bytes of one planned decode gather launch of `out_rows` output rows:
    the committed ncu summary of a small case with the same page sharing
    (each page named ~16 times) gives DRAM bytes per output row, which is
    scaled by the rows of the full launch. None when the summary is missing
    or the kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        text = open(path).read()
    except OSError:
        return None
    src_hash = per_row = None
    for line in text.splitlines():
        if line.startswith("kernel_sources_sha256_16:"):
            src_hash = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_output_row:"):
            per_row = float(line.split(":", 1)[1].strip())
    if per_row is None or src_hash != sources_hash(sources):
        return None
    return round(per_row * out_rows)


# ------------------------------------------------------------------ CPU oracle

def cpu_model() -> str:
    """Host CPU name, best effort (x86 'model name', Arm implementer/part)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    for line in info.splitlines():
        if line.lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    parts = {ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU part")}
    impl = {ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU implementer")}
    known = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd0c": "Arm Neoverse-N1"}
    return ", ".join(sorted(known.get(p, f"implementer {','.join(sorted(impl))} part {p}") for p in parts)) or "unknown"


def oracle_sample(budget_s: float = 12.0, threads: int = 1):
    """The oracle, as it stands, on a bounded sample of the step, repeated
    until `budget_s` has elapsed. One sample: a 257-page pool of the same
    model shape; translate 512 slots; the 256-token all-layer store; 256
    decode tokens stored for one layer; 16 sequences x 4096 tokens gathered
    for one layer, each through a permutation of the 256 allocatable pages
    (so each page is named 16 times, as in the step); 512 moved tokens. Rates
    count method bytes, as the GPU line does. With threads > 1 the sample is split
    across threads (gather by sequence, all-layer store by layer, the rest by
    token ranges), all on one shared pool mirror with disjoint writes; the
    oracle's C routines release the GIL."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle as ora

    P, n_seq = 257, 16  # 16 sequences x 256 pages of 256: each page named 16 times, as in the step
    sh = SHAPE.scaled(P)
    L = sh.layer_num
    o = ora.Oracle(ora.Geometry(L, sh.head_num, sh.head_dim, sh.itemsize, sh.page_size, P))
    M = synth.sentinel_bytes(5, 0, o.raw_bytes())
    rng = synth.rng_for(sh.seed, synth.S_MISC, 1)
    ps, R = sh.page_size, sh.row_bytes
    slots = synth.distinct_slots(rng, ps, P * ps, 256 + 256 + 1024)
    bt = np.stack([1 + rng.permutation(P - 1)[:CTX // ps] for _ in range(n_seq)]).astype(np.int32)
    kc, vc = synth.kv_pair(sh, L * 256, 1)
    kc, vc = kc.reshape(L, 256, -1), vc.reshape(L, 256, -1)
    kd, vd = synth.kv_pair(sh, 256, 0)
    src, _ = o.translate(slots[512:1024])
    dst, _ = o.translate(slots[1024:])
    outk = np.empty((n_seq * CTX, R), np.uint8)
    outv = np.empty((n_seq * CTX, R), np.uint8)
    g_all = synth.GatherBatch(bt, np.zeros(n_seq, np.int32), np.full(n_seq, CTX, np.int32))
    per, gb = step_bytes(g_all, sh, n_decode=256, n_chunk=256, n_move=512)
    per_rep = per["translate"] + per["store_all_layers"] + per["store_layer"] // L + gb["method"] + per["move"]

    def rng_of(n, w):
        k = -(-n // threads)
        return slice(min(n, w * k), min(n, (w + 1) * k))

    def work(w):
        a = rng_of(512, w)
        o.translate(slots[:512][a])
        for layer in range(w, L, threads):  # all-layer store, split by layer
            o.store(M, layer, slots[256:512], kc[layer], vc[layer])
        d = rng_of(256, w)
        o.store(M, 5, slots[:256][d], kd[d], vd[d])
        sq = rng_of(n_seq, w)
        g = synth.GatherBatch(bt[sq], np.zeros(sq.stop - sq.start, np.int32),
                              np.full(sq.stop - sq.start, CTX, np.int32))
        r0 = sq.start * CTX
        o.gather(M, 5, g.block_table, g.seq_len, g.cu + r0, g.seq_start, n_seq * CTX, outk, outv)
        m = rng_of(512, w)
        o.move(M, src[m], dst[m])

    t0 = time.perf_counter()
    reps = 0
    with ThreadPoolExecutor(max_workers=threads) as ex:
        while True:
            list(ex.map(work, range(threads)))
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    return {"value": per_rep * reps / el / GB, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": (f"{reps} reps on {threads} thread(s) of: a 257-page pool of the same shape; translate 512 "
                       f"slots; store_all 256 tokens x 32 layers; store_layer 256 tokens; gather {n_seq} seqs x 4096 "
                       f"tokens for one layer (each table a permutation of pages 1..256: each page named 16 times); "
                       f"move 512 tokens; method bytes; {el:.1f} s"),
            "cpu_model": cpu_model(), "seconds": el}


# ------------------------------------------------------------------ ranks

def reduce_max(values, device=None):
    """Max over ranks of per-rank timings (identity when not distributed).
    Every rank gets the result; rank 0 prints it."""
    import torch
    import torch.distributed as dist

    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_gbps(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """Weak scaling: every rank moves its own step's bytes; the job's rate is
    all ranks' bytes over the slowest rank's time."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / GB


# ------------------------------------------------------------------ GPU arm

class Step:
    """The timed step's device state and launch sequence (see make_step)."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def virtual_tables(g: synth.GatherBatch, num_pages: int, seed: int = 77):
    """The same block tables as virtual pages: a random bijection v2p of pages
    1..P-1 (page 0, the sink, maps to itself) and, per entry, the virtual
    page that v2p maps to the table's physical page. Returns (virt, v2p)."""
    rng = np.random.default_rng(seed)
    v2p = np.zeros(num_pages, np.int32)
    v2p[1:] = 1 + rng.permutation(num_pages - 1)
    inv = np.zeros(num_pages, np.int32)
    inv[v2p] = np.arange(num_pages, dtype=np.int32)
    virt = np.where(g.block_table < 0, -1, inv[np.maximum(g.block_table, 0)]).astype(np.int32)
    return virt, v2p


def make_step(gt, pool, inp, dev, stream, kernel_facing: bool = False) -> Step:
    """Device buffers of one rank's inputs and the step that bench.py times:
    translate -> all-layer store of the chunk -> gather plan -> 32 x (decode
    store + planned gather) -> move, every call on `stream`. The move's ids
    are kernel-facing, translated once here with the library. The gather
    output buffers are shared by the layers (the last layer's rows remain).
    With kernel_facing the tables arrive as virtual pages with a page map:
    the step first builds the prefix-only kernel-facing table
    (kv_translate_block_table), then plans and gathers through it
    (kv_gather_plan_kf, kv_gather_layer_planned_kf); the rows read are the
    same. Step.step(x, record, out) runs one step on the inputs x
    (Step.dev_in, or any dict of device tensors of the same shapes),
    gathering into `out` (a (K, V) pair of device tensors shaped like
    Step.out_k, default Step.out_k / Step.out_v); with record=True it
    appends CUDA events around each gather to Step.gather_ev."""
    import torch

    L, R = SHAPE.layer_num, SHAPE.row_bytes

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    g = inp["g"]
    dev_in = dict(slots=d(inp["slots"]), bt=d(g.block_table), ln=d(g.seq_len), cu=d(g.cu),
                  k_dec=d(inp["k_dec"]), v_dec=d(inp["v_dec"]), k_chunk=d(inp["k_chunk"]),
                  v_chunk=d(inp["v_chunk"]))
    kf = None
    if kernel_facing:
        virt, v2p = virtual_tables(g, SHAPE.num_pages)
        dev_in.update(virt=d(virt), v2p=d(v2p))
        kf = torch.empty_like(dev_in["bt"])
    ids = torch.empty(N_DECODE + N_CHUNK, dtype=torch.int32, device=dev)
    mv = torch.empty(2 * N_MOVE, dtype=torch.int32, device=dev)
    gt.kv_translate(pool, d(np.concatenate([inp["move_src"], inp["move_dst"]])), mv, stream=stream)
    mv_src, mv_dst = mv[:N_MOVE], mv[N_MOVE:]
    out_k = torch.empty((g.total, R), dtype=torch.uint8, device=dev)
    out_v = torch.empty_like(out_k)
    plan = torch.empty(gt.kv_gather_plan_bytes(pool, *g.block_table.shape) // 4, dtype=torch.int32, device=dev)
    gather_ev = []

    def step(x, record=False, out=None):
        ok, ov = (out_k, out_v) if out is None else out
        gt.kv_translate(pool, x["slots"], ids, stream=stream)
        gt.kv_store_all_layers(pool, ids[N_DECODE:], x["k_chunk"], x["v_chunk"], stream=stream)
        if kernel_facing:
            gt.kv_translate_block_table(pool, x["virt"], x["ln"], x["v2p"], kf, stream=stream)
            gt.kv_gather_plan_kf(pool, kf, x["ln"], plan=plan, stream=stream)
        else:
            gt.kv_gather_plan(pool, x["bt"], x["ln"], plan=plan, stream=stream)
        for layer in range(L):
            gt.kv_store_layer(pool, layer, ids[:N_DECODE], x["k_dec"][layer], x["v_dec"][layer], stream=stream)
            if record:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            if kernel_facing:
                gt.kv_gather_layer_planned_kf(pool, layer, plan, kf, x["ln"], x["cu"], ok, ov, stream=stream)
            else:
                gt.kv_gather_layer_planned(pool, layer, plan, x["bt"], x["ln"], x["cu"], ok, ov, stream=stream)
            if record:
                e1.record(stream)
                gather_ev.append((e0, e1))
        gt.kv_move(pool, mv_src, mv_dst, stream=stream)

    return Step(step=step, dev_in=dev_in, ids=ids, mv_src=mv_src, mv_dst=mv_dst, out_k=out_k, out_v=out_v,
                plan=plan, gather_ev=gather_ev, kf=kf)



TARGETS = ["store:3", "store_all:3", "move:2", "move:4"]
TARGET_NAMES = {"store:3": "store_layer, llama3-8b-prefill (32768 tokens per layer, 2 % tombstones)",
                "store_all:3": "store_all_layers, llama3-8b-prefill ([32, 32768, 8, 128] bf16, 4 GiB)",
                "move:2": "move, llama3-8b-decode pool (8192 tokens x 64 row-blocks x 2 KiB)",
                "move:4": "move, swa-fp8 pool (8192 tokens x 48 row-blocks x 512 B)"}


def run_targets(iters: int) -> dict:
    """The store and move workloads graded beside the gather, each timed per
    launch with CUDA events (mean over `iters` launches after 3 warm-ups; L2
    flushed before each launch whose working set is under 4x L2), on its own
    pool, freed afterwards."""
    ns = argparse.Namespace(iters=iters, torch_ref=0, pages=0, layers=0, seqs=0, only=",".join(TARGETS))
    out = {}
    for rec in run_micro(ns, quiet=True):
        if rec.get("micro") == "skipped":
            out[f"skipped_cfg{rec['cfg']}"] = rec["reason"]
            continue
        key = {"store_layer": "store", "store_all_layers": "store_all", "move": "move"}[rec["micro"]]
        key = f"{key}:{rec['cfg']}"
        out[key] = {"what": TARGET_NAMES[key], "us_per_call": rec["us_per_call"],
                    "method_bytes_per_call": rec["useful_bytes_per_call"], "GBps": rec["useful_GBps"],
                    "frac": round(rec["pct_of_hbm_peak"] / 100, 4), "rows_per_s": rec["rows_per_s"],
                    "calls": rec["calls"],
                    "l2_flush": rec.get("l2_flush")}
    return out


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import gather_translate_kv_gb300 as gt
    from gather_translate_kv_gb300 import build as gbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        gbuild.build()
    if world > 1:
        dist.barrier()
    gt.lib()

    sh = SHAPE
    L, ps = sh.layer_num, sh.page_size
    inp = make_inputs(rank)
    total, pad = gt.kv_pool_required_bytes(gt.make_desc(L, sh.head_num, sh.head_dim, sh.itemsize, ps,
                                                        sh.num_pages))
    raw = torch.empty(total + pad, dtype=torch.uint8, device=dev)
    synth.fill_sentinel_torch(raw, 17 + rank)
    pool = gt.kv_pool_create(gt.make_desc(L, sh.head_num, sh.head_dim, sh.itemsize, ps, sh.num_pages), raw)

    stream = torch.cuda.current_stream(dev)
    st = make_step(gt, pool, inp, dev, stream)
    step, dev_in, ids, gather_ev, g = st.step, st.dev_in, st.ids, st.gather_ev, inp["g"]
    launches_per_step = 1 + 1 + 3 + 2 * L + 1  # the plan is 3 kernels (+ a memset)

    for _ in range(args.warmup):
        step(dev_in)
    torch.cuda.synchronize(dev)
    assert gt.kv_pool_last_error(pool) == 0

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step(dev_in, record=True)
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end) / args.steps
    gather_ms = statistics.mean(a.elapsed_time(b) for a, b in gather_ev)
    dev_err = gt.kv_pool_last_error(pool)

    # end to end, through the public API: every step's inputs go from pinned
    # host memory to the device, and every step's product comes back to pinned
    # host memory: the last layer's gathered K and V (4.29 GB) and the
    # translated ids. Three forms, each over the same number of steps:
    #  pipelined  (the figure reported): two sets of device inputs and
    #             outputs; step i's upload runs on a copy stream while step
    #             i-1 computes, and its result download on a second copy
    #             stream while step i+1 computes; the device error word is
    #             read once, at the end, and every copy has landed before the
    #             clock stops
    #  serial     upload, step, download, error word, one after the other
    #  no result  as serial, without the 4.29 GB download
    host = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in
            dict(slots=inp["slots"], bt=g.block_table, ln=g.seq_len, cu=g.cu, k_dec=inp["k_dec"],
                 v_dec=inp["v_dec"], k_chunk=inp["k_chunk"], v_chunk=inp["v_chunk"]).items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    ids_host = torch.empty(ids.shape, dtype=ids.dtype).pin_memory()
    out_k_host = torch.empty(st.out_k.shape, dtype=torch.uint8).pin_memory()
    out_v_host = torch.empty(st.out_v.shape, dtype=torch.uint8).pin_memory()
    d2h_small = ids_host.numel() * 4 + 4
    d2h = d2h_small + out_k_host.numel() + out_v_host.numel()
    stages = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    outs = [(st.out_k, st.out_v), (torch.empty_like(st.out_k), torch.empty_like(st.out_v))]
    ids_sets = [torch.empty_like(ids) for _ in range(2)]  # each step's ids, kept until downloaded
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in_ready", "computed", "read")}

    def e2e_serial(read_result: bool):
        for k, v in host.items():
            stages[0][k].copy_(v, non_blocking=True)
        step(stages[0])
        ids_host.copy_(ids, non_blocking=True)
        if read_result:
            out_k_host.copy_(st.out_k, non_blocking=True)
            out_v_host.copy_(st.out_v, non_blocking=True)
        return gt.kv_pool_last_error(pool, stream)  # synchronizes: the step's result is on the host

    def e2e_pipelined(i: int):
        b = i % 2
        if i >= 2:
            s_in.wait_event(ev["computed"][b])   # step i-2 has finished reading these inputs
        with torch.cuda.stream(s_in):
            for k, v in host.items():
                stages[b][k].copy_(v, non_blocking=True)
        ev["in_ready"][b].record(s_in)
        stream.wait_event(ev["in_ready"][b])
        if i >= 2:
            stream.wait_event(ev["read"][b])     # step i-2's result has left these outputs
        step(stages[b], out=outs[b])
        ids_sets[b].copy_(ids)  # the next step's translate rewrites ids
        ev["computed"][b].record(stream)
        s_out.wait_event(ev["computed"][b])
        with torch.cuda.stream(s_out):
            ids_host.copy_(ids_sets[b], non_blocking=True)
            out_k_host.copy_(outs[b][0], non_blocking=True)
            out_v_host.copy_(outs[b][1], non_blocking=True)
        ev["read"][b].record(s_out)

    e2e_steps = max(3, args.steps // 2)
    e2e_s = {}
    bad = 0
    for form in ("serial", "no_result"):
        for _ in range(2):
            e2e_serial(form == "serial")
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            bad |= e2e_serial(form == "serial")
        barrier()
        e2e_s[form] = (time.perf_counter() - t0) / e2e_steps
    for i in range(2):
        e2e_pipelined(i)
    torch.cuda.synchronize(dev)
    barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_pipelined(i)
    bad |= gt.kv_pool_last_error(pool, stream)  # synchronizes the compute stream
    s_out.synchronize()                          # the last step's result is on the host
    barrier()
    e2e_s["pipelined"] = (time.perf_counter() - t0) / e2e_steps
    # the pipelined loop's last result is the last layer's gather of its last step
    result_ok = bool(torch.equal(out_k_host[:4096].to(dev), outs[(e2e_steps - 1) % 2][0][:4096]))

    # the same step with the read path of the pages: virtual tables and a page
    # map, the prefix-only kernel-facing table built every step, the plan and
    # the gathers reading through it (one more launch per step)
    stk = make_step(gt, pool, inp, dev, stream, kernel_facing=True)
    for _ in range(args.warmup):
        stk.step(stk.dev_in)
    barrier()
    t0k = torch.cuda.Event(enable_timing=True)
    t1k = torch.cuda.Event(enable_timing=True)
    t0k.record(stream)
    for _ in range(args.steps):
        stk.step(stk.dev_in, record=True)
    t1k.record(stream)
    barrier()
    kf_ms = t0k.elapsed_time(t1k) / args.steps
    kf_gather_ms = statistics.mean(a.elapsed_time(b) for a, b in stk.gather_ev)
    kf_ok = bool(torch.equal(stk.out_k, st.out_k) and torch.equal(stk.out_v, st.out_v))
    bad |= gt.kv_pool_last_error(pool, stream)
    del stk

    sb, gb = step_bytes(g)
    step_total = sum(sb.values())
    kf_extra = g.block_table.size * (4 + 4 + 4)  # table build: virtual entry + page map entry read, entry written
    step_rows = (L * gb["rows"] * 2 + N_CHUNK * 2 * L + L * N_DECODE * 2 + N_MOVE * 2 * L)  # K and V rows
    per_reader_total = step_total - sb["gather"] + L * gb["per_reader"]
    ms, e2e_ms, e2e_ser_ms, e2e_nr_ms, gather_ms, kf_ms, kf_gather_ms = reduce_max(
        [ms, e2e_s["pipelined"] * 1e3, e2e_s["serial"] * 1e3, e2e_s["no_result"] * 1e3, gather_ms, kf_ms,
         kf_gather_ms], dev)
    del stages, outs, ids_sets, host, out_k_host, out_v_host
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = measured_hbm_peak()
    achieved = gb["method"] / (gather_ms * 1e-3) / GB
    traffic = profiled_traffic(gb["rows"])
    line = {
        "metric": "KV store/gather/move useful GB/s and % of GB300 HBM peak (byte-exact vs oracle)",
        "value": round(whole_job_gbps(step_total, world, ms), 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u8",
        "data": "synthetic (seeded: bf16 N(0,1) K/V, random block tables and slots)",
        "config": {"workload": WORKLOAD, "kv_dtype": "bf16",
                   "useful_bytes": "method bytes: each distinct source row read once, each output row "
                                   "written once, plus index bytes",
                   "useful_bytes_per_step": step_total, "useful_bytes_by_kernel": sb,
                   "gather_per_launch": gb,
                   "l2": "no flush: inputs larger than L2 (8 GiB pool, 4 GiB gather output per layer)",
                   "parallelism": f"replicas x{world}",
                   "pct_of_hbm_peak": round(100 * step_total / (ms * 1e-3) / GB / peak, 1),
                   # rows copied per second: the gathers' output rows, the stores' and the move's rows
                   "rows_per_s": round(world * step_rows / (ms * 1e-3), 1),
                   # every output row's source counted once per sequence that reads it; L2 serves the
                   # repeats, so this rate is not bounded by the HBM peak
                   "effective_GBps_per_reader": round(whole_job_gbps(per_reader_total, world, ms), 1),
                   "useful_bytes_per_output_reference": per_reader_total},
        "roofline": {"bound": "hbm", "kernel": "kv_gather_layer_planned (k_gather_fan<true, false>)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes_per_launch": gb["method"],
                     "avg_launch_ms": round(gather_ms, 4),
                     "dram_achieved": None if traffic is None else round(traffic / (gather_ms * 1e-3) / GB, 1),
                     "dram_frac": None if traffic is None else round(traffic / (gather_ms * 1e-3) / GB / peak, 4)},
        "e2e": {"value": round(whole_job_gbps(step_total, world, e2e_ms), 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h - 4, "ms_per_step": round(e2e_ms, 3),
                "steps": e2e_steps, "result_matches_device": result_ok,
                "result": "every step: the last layer's gathered K and V and the translated ids; the device "
                          "error word once at the end",
                "form": "pipelined: uploads and result downloads on two copy streams, overlapping the "
                        "neighbouring steps' compute (two sets of device inputs and outputs)",
                "serial": {"value": round(whole_job_gbps(step_total, world, e2e_ser_ms), 1),
                           "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ser_ms, 3)},
                "without_result_readback": {"value": round(whole_job_gbps(step_total, world, e2e_nr_ms), 1),
                                            "d2h_bytes_per_step": d2h_small, "ms_per_step": round(e2e_nr_ms, 3)}},
        "kernel_facing_read_path": {
            "what": "the same step with virtual block tables and a page map: kv_translate_block_table every "
                    "step, then kv_gather_plan_kf and kv_gather_layer_planned_kf",
            "value": round(whole_job_gbps(step_total + kf_extra, world, kf_ms), 1), "unit": "GB/s",
            "ms_per_step": round(kf_ms, 4), "gather_avg_launch_ms": round(kf_gather_ms, 4),
            "gather_frac": round(gb["method"] / (kf_gather_ms * 1e-3) / GB / measured_hbm_peak()[0], 4),
            "output_equals_physical_table_step": kf_ok, "steps": args.steps},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "device_errors": dev_err | bad,
    }
    # the graded store and move workloads, after the step's pool is gone
    del st, dev_in, ids, gather_ev
    gt.kv_pool_destroy(pool)
    del raw
    torch.cuda.empty_cache()
    if world == 1 and not args.no_targets:
        clocks = ClockSampler(uuid)
        clocks.start()
        targets = run_targets(max(20, args.target_iters))
        targets["clocks"] = clocks.stop()
        line["targets"] = targets
    if world == 1 and not args.no_cpu_baseline:
        one = oracle_sample(args.cpu_budget / 2, 1)
        ncores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        many = oracle_sample(args.cpu_budget / 2, max(1, ncores))
        many.pop("seconds", None)
        many["value_1_thread"] = round(one["value"], 3)
        line["cpu_baseline"] = many
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The oracle as the reference arm: each step is a bounded sample of the
    workload, timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    oracle.build()
    budget = max(1.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    ncores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    for _ in range(args.warmup):
        oracle_sample(budget / 4, ncores)
    vals = [oracle_sample(budget, ncores) for _ in range(args.steps)]
    v = statistics.mean(x["value"] for x in vals)
    secs = sum(x["seconds"] for x in vals)
    line = {
        "impl": "reference",
        "metric": "KV store/gather/move useful GB/s and % of GB300 HBM peak (byte-exact vs oracle)",
        "value": round(v, 3), "unit": "GB/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded)", "config": {"workload": WORKLOAD, "kv_dtype": "bf16"},
        "cpu_baseline": {"value": round(v, 3), "unit": "GB/s", "cores": ncores, "kind": "oracle",
                         "sample": vals[0]["sample"], "cpu_model": vals[0]["cpu_model"]},
        "e2e": {"value": round(v, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ per-kernel table

MICRO_DEFAULT = ["ceiling:0", "translate:2", "block_table:2", "store:2", "store_slots:2", "store_graph:2", "store_all:2",
                 "gather:2", "gather_planned:2", "move:2",
                 "translate:3", "store:3", "store_slots:3", "store_all:3", "gather:3", "gather_planned:3",
                 "translate_mapped:4", "store:4", "gather:4", "gather_planned:4", "move:4",
                 "translate:5", "store:5", "store_sorted:5", "store_slots:5", "gather:5", "gather_planned:5", "move:5", "move_sorted:5",
                 "store:6", "store_all:6", "gather:6", "gather_planned:6", "move:6"]


def _payload_torch(gen, rows: int, R: int, itemsize: int, dev):
    """Seeded synthetic K or V rows on the device: bf16 N(0,1) bits, or fp8
    e4m3 bytes uniform over the 254 non-NaN codes."""
    import torch

    if itemsize == 2:
        return torch.randn((rows, R // 2), generator=gen, device=dev, dtype=torch.float32) \
            .to(torch.bfloat16).view(torch.uint8).reshape(rows, R)
    x = torch.randint(0, 254, (rows, R), generator=gen, device=dev, dtype=torch.int16)
    x += (x >= 0x7F).to(torch.int16)
    return x.to(torch.uint8)


def run_micro(args, quiet: bool = False) -> list[dict]:
    """Each kernel on each workload of the build plan, timed per launch with
    CUDA events (median), L2 flushed between launches whose working set is
    under 4x the L2 size (a 2x-L2 write followed by a 2x-L2 read, so the
    launch finds neither its data nor dirty lines in L2). One JSON line per
    (kernel, workload), printed unless `quiet`; the records are returned."""
    import torch

    import gather_translate_kv_gb300 as gt
    from gather_translate_kv_gb300 import build as gbuild

    gbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, peak_kind = measured_hbm_peak()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    flush_read = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one: the timed
        # launch starts with none of its data cached and no dirty lines left
        # for it to write back
        flush_buf.zero_()
        flush_read.max()
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    records: list[dict] = []

    def emit(line):
        records.append(line)
        if not quiet:
            print(json.dumps(line), flush=True)
    stream = torch.cuda.current_stream(dev)
    todo = args.only.split(",") if args.only else MICRO_DEFAULT
    by_cfg: dict[int, list[str]] = {}
    for item in todo:
        k, c = item.split(":")
        by_cfg.setdefault(int(c), []).append(k)

    def timed(fn, calls: int, flush: bool):
        ms = []
        for i in range(calls + 3):
            if flush:
                flush_l2()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(i)
            e1.record(stream)
            e1.synchronize()
            if i >= 3:
                ms.append(e0.elapsed_time(e1))
        return ms

    def report(kernel, cfg, workload, ms, useful, rows, extra=None, ref_ms=None):
        # the event clock ticks in ~2 us steps on this part: the mean over many
        # launches resolves short kernels better than the median
        med = statistics.mean(ms)
        line = {"micro": kernel, "cfg": cfg, "workload": workload, "calls": len(ms),
                "us_per_call": round(med * 1e3, 2), "us_median": round(statistics.median(ms) * 1e3, 2),
                "useful_bytes_per_call": useful,
                "useful_GBps": round(useful / (med * 1e-3) / GB, 1),
                "pct_of_hbm_peak": round(100 * useful / (med * 1e-3) / GB / peak, 1),
                "rows_per_s": round(rows / (med * 1e-3), 1), "peak_GBps": peak, "peak_source": peak_kind}
        if ref_ms:
            r = statistics.mean(ref_ms)
            line["torch_indexing_us"] = round(r * 1e3, 2)
            line["speedup_vs_torch_indexing"] = round(r / med, 2)
        line.update(extra or {})
        emit(line)

    if "ceiling" in by_cfg.pop(0, []):
        # context for the HBM-bound kernels: torch's own fill, copy and
        # reduction over 4 GiB (library kernels, not part of the path), i.e.
        # what a write-only, a copy and a read-only stream reach on this GPU
        nb = 4 << 30
        a = torch.empty(nb, dtype=torch.uint8, device=dev)
        b = torch.empty(nb, dtype=torch.uint8, device=dev)
        a.fill_(1)
        w = a.view(torch.int32)
        b64 = b.view(torch.int64)
        ms = timed(lambda i: b64.fill_(i), args.iters, False)
        report("ceiling_write", 0, "4 GiB, torch fill_ of int64 (write only)", ms, nb, nb // 16)
        ms = timed(lambda i: b.zero_(), args.iters, False)
        report("ceiling_write_zero", 0, "4 GiB, torch zero_ (write only)", ms, nb, nb // 16)
        ms = timed(lambda i: b.copy_(a), args.iters, False)
        report("ceiling_copy", 0, "4 GiB, torch copy_ (read + write)", ms, 2 * nb, nb // 16)
        ms = timed(lambda i: w.amax(), args.iters, False)
        report("ceiling_read", 0, "4 GiB, torch amax (read only)", ms, nb, nb // 16)
        del a, b, w, b64
        torch.cuda.empty_cache()

    for cfg, kernels in sorted(by_cfg.items()):
        sh = synth.SHAPES[cfg]
        if args.pages or args.layers:
            sh = synth.Shape(cfg, sh.name + "-small", args.layers or sh.layer_num, sh.head_num, sh.head_dim,
                             sh.itemsize, sh.page_size, args.pages or sh.num_pages, sh.latent)
        L, R, ps, P = sh.layer_num, sh.row_bytes, sh.page_size, sh.num_pages
        kvr = 1 if sh.latent else 2  # rows per layer per token (MLA: one latent row, no V)
        desc = gt.make_desc(L, sh.head_num, sh.head_dim, sh.itemsize, ps, P, latent_only=sh.latent)
        total, pad = gt.kv_pool_required_bytes(desc)
        free, _ = torch.cuda.mem_get_info(dev)
        if total + pad + (8 << 30) > free:
            emit({"micro": "skipped", "cfg": cfg, "reason": f"{free / 2**30:.1f} GiB free"})
            continue
        raw = torch.empty(total + pad, dtype=torch.uint8, device=dev)
        synth.fill_sentinel_torch(raw, 99)
        pool = gt.kv_pool_create(desc, raw)

        def d(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

        # The report's own method on the same bytes, for comparison: dense
        # per-layer views over the raw buffer (build_mha_views: block b starts
        # at b*ps*R, rows of R bytes) and torch indexing through them.
        n_rows_view = P * kvr * L * ps

        def view(block):
            return torch.as_strided(raw, size=(n_rows_view, R), stride=(R, 1), storage_offset=block * ps * R)

        slots = synth.store_slots(sh, 0)
        n = slots.size
        n_tomb = int(np.count_nonzero(slots < 0))
        slots_d = d(slots)
        ids = torch.empty(n, dtype=torch.int32, device=dev)
        gt.kv_translate(pool, slots_d, ids)
        calls = args.iters
        if "translate" in kernels:
            ms = timed(lambda i: gt.kv_translate(pool, slots_d, ids), calls, True)
            report("translate", cfg, f"{n} slots", ms, n * 12, n)
        if "translate_mapped" in kernels:
            # a hybrid model's SWA layers: full-pool slots through a full -> SWA
            # token map over 4x this pool's slots, a quarter of it cleared
            rm = np.random.default_rng(5)
            n_full = 4 * P * ps
            tmap = rm.integers(0, P * ps, size=n_full).astype(np.int64)
            tmap[rm.random(n_full) < 0.25] = -1
            fslots = d(rm.integers(0, n_full, size=n).astype(np.int64))
            tmap_d = d(tmap)
            ms = timed(lambda i: gt.kv_translate_mapped(pool, fslots, ids, tmap_d), calls, True)
            report("translate_mapped", cfg, f"{n} slots through a {n_full}-entry token map", ms, n * 20, n)
            gt.kv_translate(pool, slots_d, ids)
        if "block_table" in kernels:
            gbt = synth.gather_batch(sh)
            vt = d(gbt.block_table)
            vmap = d(np.random.default_rng(3).permutation(P).astype(np.int32))
            kf = torch.empty_like(vt)
            lnt = d(gbt.seq_len)
            ne = gbt.block_table.size
            ms = timed(lambda i: gt.kv_translate_block_table(pool, vt, lnt, vmap, kf), calls, True)
            report("translate_block_table", cfg, f"{gbt.block_table.shape[0]} x {gbt.block_table.shape[1]} entries",
                   ms, ne * 12, ne)
        if "store" in kernels or "store_graph" in kernels or "store_slots" in kernels or "store_sorted" in kernels:
            K = _payload_torch(gen, n, R, sh.itemsize, dev)
            V = None if sh.latent else _payload_torch(gen, n, R, sh.itemsize, dev)
            useful = (n - n_tomb) * 2 * kvr * R + n * 4
            flush = useful < 4 * l2
            if "store" in kernels:
                ms = timed(lambda i: gt.kv_store_layer(pool, i % L, ids, K, V), max(calls, L), flush)
                ids64 = ids.to(torch.int64)

                def ref_store(i):
                    view(kvr * (i % L))[ids64] = K
                    if V is not None:
                        view(kvr * (i % L) + 1)[ids64] = V
                ref = timed(ref_store, max(calls, L), flush) if args.torch_ref else None
                report("store_layer", cfg, f"{n} tokens per layer ({n_tomb} tombstones)", ms, useful, 2 * n,
                       {"l2_flush": flush, "tombstone_bytes": n_tomb * 4 * R}, ref)
            if "store_sorted" in kernels:
                # the same tokens in destination order, their K/V rows permuted alike (done here,
                # outside the timing): how much of the store's time is where its rows land
                order = torch.argsort(ids)
                ids_s = ids[order].contiguous()
                K_s = K[order].contiguous()
                V_s = None if V is None else V[order].contiguous()
                ms = timed(lambda i: gt.kv_store_layer(pool, i % L, ids_s, K_s, V_s), max(calls, L), flush)
                report("store_layer_sorted", cfg, f"{n} tokens per layer in destination order ({n_tomb} tombstones)",
                       ms, useful, 2 * n, {"l2_flush": flush})
                del ids_s, K_s, V_s
            if "store_slots" in kernels:
                ms = timed(lambda i: gt.kv_store_layer_slots(pool, i % L, slots_d, K, V), max(calls, L), flush)
                report("store_layer_slots", cfg, f"{n} slots per layer, translate fused ({n_tomb} tombstones)",
                       ms, useful + n * 4, 2 * n, {"l2_flush": flush})
            if "store_graph" in kernels:
                g = torch.cuda.CUDAGraph()
                s2 = torch.cuda.Stream(dev)
                s2.wait_stream(stream)
                with torch.cuda.stream(s2):
                    for layer in range(L):
                        gt.kv_store_layer(pool, layer, ids, K, V)
                stream.wait_stream(s2)
                with torch.cuda.graph(g):
                    for layer in range(L):
                        gt.kv_store_layer(pool, layer, ids, K, V)
                ms = timed(lambda i: g.replay(), calls, L * useful < 4 * l2)
                report("store_layer_x32_graph", cfg, f"{L} per-layer stores of {n} tokens in one CUDA graph",
                       ms, L * useful, 2 * n * L, {"l2_flush": L * useful < 4 * l2})
                del g
            del K, V
        if "store_all" in kernels:
            na = n if cfg not in (2, 6) else 256
            Ka = _payload_torch(gen, L * na, R, sh.itemsize, dev)
            Va = None if sh.latent else _payload_torch(gen, L * na, R, sh.itemsize, dev)
            ta = int(np.count_nonzero(slots[:na] < 0))
            useful = L * (na - ta) * 2 * kvr * R + na * 4
            flush = useful < 4 * l2
            ms = timed(lambda i: gt.kv_store_all_layers(pool, ids[:na], Ka, Va), calls, flush)
            report("store_all_layers", cfg, f"{na} tokens x {L} layers", ms, useful, 2 * L * na,
                   {"l2_flush": flush})
            del Ka, Va
        if "gather" in kernels or "gather_planned" in kernels:
            gb = synth.gather_batch(sh) if not args.seqs else synth.GatherBatch(
                synth.gather_batch(sh).block_table[: args.seqs], np.zeros(args.seqs, np.int32),
                synth.gather_batch(sh).seq_len[: args.seqs])
            rows = gb.total
            ok = torch.empty((rows, R), dtype=torch.uint8, device=dev)
            ov = None if sh.latent else torch.empty_like(ok)
            bt, ln, cu, st = d(gb.block_table), d(gb.seq_len), d(gb.cu), d(gb.seq_start)
            acct = gather_bytes(gb, ps, R, kvr)
            useful = acct["method"]  # distinct source rows once, output rows once, index bytes
            flush = acct["per_reader"] < 4 * l2
            layers = list(range(L)) if cfg != 5 else [0, L - 1]
            distinct = len(np.unique(gb.block_table))
            share = {"l2_flush": flush, "distinct_pages": distinct,
                     "page_reads_per_distinct_page": round(gb.block_table.size / max(1, distinct), 2),
                     "per_reader_bytes_per_call": acct["per_reader"]}
            if "gather_planned" in kernels:
                plan = gt.kv_gather_plan(pool, bt, ln, st)
                ms = timed(lambda i: gt.kv_gather_layer_planned(pool, layers[i % len(layers)], plan, bt, ln, cu, ok,
                                                                ov, st), max(calls, len(layers)), flush)
                msp = timed(lambda i: gt.kv_gather_plan(pool, bt, ln, st, plan=plan), calls, True)
                extra = dict(share, plan_build_us=round(statistics.mean(msp) * 1e3, 2))
                if P <= 65536:  # the allocation-free plan's fixed workspace
                    msn = timed(lambda i: gt.kv_gather_plan_noalloc(pool, bt, ln, plan, st), calls, True)
                    extra["plan_build_noalloc_us"] = round(statistics.mean(msn) * 1e3, 2)
                report("gather_layer_planned", cfg, f"{gb.block_table.shape[0]} seqs, {rows} rows, page-major plan",
                       ms, useful, rows, extra)
            ms = None
            if "gather" in kernels:
                ms = timed(lambda i: gt.kv_gather_layer(pool, layers[i % len(layers)], bt, ln, cu, ok, ov, st),
                           max(calls, len(layers)), flush)
            ref = None
            if args.torch_ref and ms is not None:
                # view rows of every output token, precomputed (not timed)
                seq = np.repeat(np.arange(gb.block_table.shape[0]), gb.seq_len - gb.seq_start)
                j = np.concatenate([np.arange(a, b) for a, b in zip(gb.seq_start, gb.seq_len)])
                vrow = torch.from_numpy(gb.block_table[seq, j // ps].astype(np.int64) * (kvr * L * ps) + j % ps).to(dev)

                def ref_gather(i):
                    layer = layers[i % len(layers)]
                    torch.index_select(view(kvr * layer), 0, vrow, out=ok)
                    if ov is not None:
                        torch.index_select(view(kvr * layer + 1), 0, vrow, out=ov)
                ref = timed(ref_gather, max(calls, len(layers)), flush)
            if ms is not None:
                report("gather_layer", cfg, f"{gb.block_table.shape[0]} seqs, {rows} rows", ms, useful, rows, share,
                       ref)
            del ok, ov
        if "move" in kernels or "move_sorted" in kernels:
            src, dst = synth.move_slots(sh)
            m = src.size
            mv = torch.empty(2 * m, dtype=torch.int32, device=dev)
            gt.kv_translate(pool, d(np.concatenate([src, dst])), mv)
            useful = m * (kvr * L * R * 2 + 8)
            flush = useful < 4 * l2
            if "move_sorted" in kernels:  # the same pairs in destination order (sorted outside the timing)
                order = torch.argsort(mv[m:])
                ms_s, md_s = mv[:m][order].contiguous(), mv[m:][order].contiguous()
                ms = timed(lambda i: gt.kv_move(pool, ms_s, md_s), calls, flush)
                report("move_sorted", cfg, f"{m} tokens x {kvr * L} row-blocks in destination order", ms, useful,
                       kvr * L * m, {"l2_flush": flush})
            if "move" in kernels:
                ms = timed(lambda i: gt.kv_move(pool, mv[:m], mv[m:]), calls, flush)
                ref = None
                if args.torch_ref:
                    s64, d64 = mv[:m].to(torch.int64), mv[m:].to(torch.int64)

                    def ref_move(i):  # every layer's K and V view, one indexing op each
                        for b in range(kvr * L):
                            vb = view(b)
                            vb[d64] = vb[s64]
                    ref = timed(ref_move, max(3, calls // 4), flush)
                report("move", cfg, f"{m} tokens x {kvr * L} row-blocks", ms, useful, kvr * L * m,
                       {"l2_flush": flush}, ref)
        err = gt.kv_pool_last_error(pool)
        assert err == 0, f"device error bits {err}"
        gt.kv_pool_destroy(pool)
        del raw
        torch.cuda.empty_cache()
    del flush_buf, flush_read
    torch.cuda.empty_cache()
    return records


# ------------------------------------------------------------------ CPU baseline table

CPU_TABLE = {  # cfg: (oracle pool pages, store tokens, gather seqs, gather pages per seq, window, move pairs)
    1: (64, 100, 1, 8, None, 20),
    2: (64, 256, 16, 63, None, 256),
    3: (32, 1984, 1, 31, None, 0),
    4: (256, 512, 50, 5, 128, 512),
    5: (64, 14000, 64, 4, None, 512),
}
CPU_KERNELS = ("translate", "store_layer", "store_all_layers", "gather_layer", "move")


def _cpu_cases(cfg: int):
    """Oracle inputs for one workload, on a pool of the workload's model shape
    with fewer pages (the full pools are 8 to 119 GiB): tokens at distinct
    random slots outside page 0 (no tombstones, so that threads write disjoint
    rows), K/V bytes, block tables whose sequences take random distinct pages,
    and disjoint move pairs."""
    import oracle as ora

    sh = synth.SHAPES[cfg]
    P, n, S_, npg, win, m = CPU_TABLE[cfg]
    sh = sh.scaled(P)
    ps, R, L = sh.page_size, sh.row_bytes, sh.layer_num
    o = ora.Oracle(ora.Geometry(L, sh.head_num, sh.head_dim, sh.itemsize, ps, P))
    rng = synth.rng_for(sh.seed, synth.S_MISC, 11)
    slots = synth.distinct_slots(rng, ps, P * ps, n + 2 * m)
    K = rng.integers(0, 256, size=(L, n, R), dtype=np.uint8)
    V = rng.integers(0, 256, size=(L, n, R), dtype=np.uint8)
    bt = np.stack([1 + rng.permutation(P - 1)[:npg] for _ in range(S_)]).astype(np.int32)
    if win is None:
        st = np.zeros(S_, np.int32)
        ln = np.full(S_, npg * ps, np.int32)
    else:
        ln = (win + rng.integers(0, npg * ps - win + 1, size=S_)).astype(np.int32)
        st = (ln - win).astype(np.int32)
    g = synth.GatherBatch(bt, st, ln)
    ids, _ = o.translate(slots[n:])
    return dict(sh=sh, o=o, slots=slots[:n], K=K, V=V, g=g, src=ids[:m], dst=ids[m:], m=m, n=n)


def _time_cpu(fn, units: int, threads: int, budget_s: float) -> float:
    """Seconds per pass of fn over `units` units split in `threads` ranges."""
    from concurrent.futures import ThreadPoolExecutor

    def ranges():
        k = -(-units // threads)
        return [(w * k, min(units, (w + 1) * k)) for w in range(threads) if w * k < units]

    parts = ranges()
    reps = 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        while True:
            list(ex.map(lambda r: fn(*r), parts))
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                return el / reps


def run_cpu_table(args):
    """The oracle, as it stands, per kernel and per workload, on one host
    thread and on every host thread, in method bytes per second (the bytes
    the GPU rows count). With a GPU, the library's --micro rate for the same
    kernel and workload is printed beside it. One JSON line per cell, then a
    markdown table."""
    import oracle as ora

    ora.build()
    ncores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    gpu = {}
    if not args.no_gpu:
        try:
            import torch

            if torch.cuda.is_available():
                items = [f"{k}:{c}" for c in CPU_TABLE for k in ("translate", "store", "store_all", "gather", "move")
                         if not (k == "move" and CPU_TABLE[c][5] == 0)]
                ns = argparse.Namespace(iters=args.iters, torch_ref=0, pages=0, layers=0, seqs=0, only=",".join(items))
                for rec in run_micro(ns, quiet=True):
                    if rec.get("micro") != "skipped":
                        gpu[(rec["micro"], rec["cfg"])] = rec
        except Exception as e:  # the table is still useful without the GPU column
            print(json.dumps({"cpu_table": "gpu column skipped", "why": repr(e)[:200]}), flush=True)
    rows = []
    for cfg in sorted(CPU_TABLE):
        c = _cpu_cases(cfg)
        o, sh, n, m, g = c["o"], c["sh"], c["n"], c["m"], c["g"]
        L, R, ps = sh.layer_num, sh.row_bytes, sh.page_size
        M = synth.sentinel_bytes(3, 0, o.raw_bytes())
        outk = np.empty((g.total, R), np.uint8)
        outv = np.empty((g.total, R), np.uint8)
        gacct = gather_bytes(g, ps, R)

        def translate(a, b):
            o.translate(c["slots"][a:b])

        def store(a, b):
            o.store(M, L - 1, c["slots"][a:b], c["K"][0, a:b], c["V"][0, a:b])

        def store_all(a, b):
            for layer in range(a, b):
                o.store(M, layer, c["slots"], c["K"][layer], c["V"][layer])

        def gather(a, b):
            sub = synth.GatherBatch(g.block_table[a:b], g.seq_start[a:b], g.seq_len[a:b])
            o.gather(M, L - 1, sub.block_table, sub.seq_len, sub.cu + g.cu[a], sub.seq_start, g.total, outk, outv)

        def move(a, b):
            o.move(M, c["src"][a:b], c["dst"][a:b])

        cases = [("translate", translate, n, n * 12), ("store_layer", store, n, n * (4 * R + 4)),
                 ("store_all_layers", store_all, L, L * n * 4 * R + n * 4),
                 ("gather_layer", gather, g.block_table.shape[0], gacct["method"])]
        if m:
            cases.append(("move", move, m, m * (2 * L * R * 2 + 8)))
        for name, fn, units, nbytes in cases:
            t1 = _time_cpu(fn, units, 1, args.cpu_cell_s)
            tn = _time_cpu(fn, units, ncores, args.cpu_cell_s)
            rec = {"cpu_table": name, "cfg": cfg, "oracle_pool_pages": sh.num_pages, "units": units,
                   "method_bytes": nbytes, "cpu_1t_GBps": round(nbytes / t1 / GB, 3),
                   "cpu_nt_GBps": round(nbytes / tn / GB, 3), "threads": ncores, "cpu_model": cpu_model()}
            if (name, cfg) in gpu:  # the same kernel in table order, as the oracle runs it
                rec["gpu_GBps"] = gpu[(name, cfg)]["useful_GBps"]
                rec["gpu_pct_of_hbm_peak"] = gpu[(name, cfg)]["pct_of_hbm_peak"]
            print(json.dumps(rec), flush=True)
            rows.append(rec)
    print()
    print(f"| Kernel | Config | GPU useful GB/s | % HBM peak | CPU 1-thread GB/s | CPU {ncores}-thread GB/s |")
    print("|---|---|---|---|---|---|")
    for r in rows:
        gp = r.get("gpu_GBps")
        print(f"| {r['cpu_table']} | {r['cfg']} | {gp if gp is not None else '-'} | "
              f"{r.get('gpu_pct_of_hbm_peak', '-')} | {r['cpu_1t_GBps']} | {r['cpu_nt_GBps']} |")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-targets", action="store_true", help="skip the store / move target workloads")
    ap.add_argument("--target-iters", type=int, default=20)
    ap.add_argument("--micro", action="store_true", help="per-kernel table instead of the step")
    ap.add_argument("--only", default="", help="micro entries, e.g. gather:2,move:4")
    ap.add_argument("--iters", type=int, default=50)
    ap.add_argument("--torch-ref", type=int, default=1, help="micro: also time torch indexing through dense views")
    ap.add_argument("--pages", type=int, default=0, help="micro: override the page count")
    ap.add_argument("--layers", type=int, default=0, help="micro: override the layer count")
    ap.add_argument("--seqs", type=int, default=0, help="micro: gather only the first N sequences")
    ap.add_argument("--cpu-table", action="store_true", help="the oracle per kernel and workload (CPU baseline)")
    ap.add_argument("--cpu-cell-s", type=float, default=0.6, help="cpu-table: seconds per cell and thread count")
    ap.add_argument("--no-gpu", action="store_true", help="cpu-table: leave out the GPU column")
    args = ap.parse_args()
    if args.cpu_table:
        run_cpu_table(args)
        return
    if args.micro:
        run_micro(args)
        return
    if args.warmup < 3 and args.impl != "reference":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
