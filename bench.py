"""Benchmark of the paged decode hot path: one step = the cache write of the
batch's new tokens followed by paged decode attention over every sequence.

Default workload: the Llama 3.1 8B-shaped single-layer decode (batch 64, 32
query / 8 KV heads, head_dim 128, bf16, 16-token blocks, contexts uniform in
[128, 2048], blocks scattered over a pool 1.25x the need) with the cache write
of the 64 new tokens.  Inputs are synthetic (paged_kv_cache_283_gb300.inputs).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload {2,3,4,5}] [--attn {auto,decode,splitk}]

Prints one JSON line.  ``value`` is achieved HBM GB/s of the whole step
(algorithmic bytes: K/V of every context token read once, q/out, block
tables, the new tokens' K/V read and written) over the device time of K
steps, replayed as CUDA graphs with inputs resident in HBM and the pool
rotated over replicas so that no step finds its K/V in L2.  ``roofline``
reports the dominant kernel alone; ``e2e`` the same metric through the
public API with host buffers and the copies inside the timed region;
``cpu_baseline`` the float64 CPU oracle on the host's cores (with a one-core
run beside it).

``--impl reference`` times the CPU oracle (the only reference this method
has) on the same workload and prints the same line with "impl": "reference".
Under torchrun (N > 1) every rank runs its own batch (weak scaling, no
collective on the data path); rank 0 prints.
"""
import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode-attention achieved HBM GB/s (frac of ~8 TB/s) and seq-layers/s"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal, context only
E2E_MIN_SECONDS = 0.25    # shortest end-to-end timed window
# --step shared-prefix: the prefix's tensor-core partitions (tokens) and the
# split-K partition size of the rest of each context
SHARED_PREFIX_SPLIT = 256
SHARED_PREFIX_PARTITION = 512


# ---------------------------------------------------------------------------
# algorithmic bytes (what one step must move at least once)

# entry-point name suffix per KV cache element type
KV_SUFFIX = {"bf16": "", "int8": "_int8", "fp8": "_fp8"}


def decode_bytes(ctx, num_seqs, hq, hkv, d, bs, kv_dtype="bf16"):
    """K/V of every attended token + q + out + block-table entries + lengths
    (an INT8 cache stores d codes and one fp32 scale per token and KV head)."""
    import numpy as np
    ctx = np.asarray(ctx, dtype=np.int64)
    per = (d + 4) if kv_dtype in ("int8", "fp8") else 2 * d
    kv = int(ctx.sum()) * hkv * per * 2
    qo = 2 * num_seqs * hq * d * 2
    tables = 4 * int((-(-ctx // bs)).sum()) + 4 * num_seqs
    return kv + qo + tables


def unique_decode_bytes(w, kv_dtype="bf16"):
    """decode_bytes with every cached token counted once however many block
    tables point at it: differs from decode_bytes only for the shared-prefix
    workload, whose 1024-token prefix is one set of blocks read by every
    sequence (logically once per sequence, from DRAM at least once)."""
    import numpy as np
    if not w.prefix_len:
        return decode_bytes(w.context_lens, w.num_seqs, w.num_q_heads, w.num_kv_heads,
                            w.head_dim, w.block_size, kv_dtype)
    per = (w.head_dim + 4) if kv_dtype in ("int8", "fp8") else 2 * w.head_dim
    tokens = w.prefix_len + int((w.context_lens.astype(np.int64) - w.prefix_len).sum())
    kv = tokens * w.num_kv_heads * per * 2
    qo = 2 * w.num_seqs * w.num_q_heads * w.head_dim * 2
    tables = 4 * int((-(-w.context_lens.astype(np.int64) // w.block_size)).sum()) + 4 * w.num_seqs
    return kv + qo + tables


def cache_write_bytes(num_tokens, hkv, d, kv_dtype="bf16"):
    """Read the new tokens' K and V, write them into the pool, read the slots."""
    written = (d + 4) if kv_dtype in ("int8", "fp8") else 2 * d
    return 2 * num_tokens * hkv * (2 * d + written) + 8 * num_tokens


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        window = [r for r in rows if t0 <= r[0] <= t1]
        used = "timed region"
        if not window:
            window = rows
            used = "whole run (timed region shorter than the sampling period)"
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = sorted(float(p[1]) for _, p in window if p[1].replace(".", "").isdigit())
        mx = max((float(p[2]) for _, p in window if p[2].replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, p in window for n, v in zip(names, p[5:9]) if v == "Active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(window), "window": used}


# ---------------------------------------------------------------------------
# CPU oracle timing (runs in a fresh process: no CUDA, one BLAS thread)

def oracle_step_sample(idx, max_seconds, out_json=True, kv="bf16"):
    """Times the float64 oracle on a bounded sample of the workload's step.

    The sample is the first n sequences of the batch (cache write of their
    new tokens + their decode), n grown until one sample takes >= 0.2 s or
    covers the batch; repeated until ``max_seconds`` have passed.  With
    ``kv="int8"`` the oracle's INT8 cache write and decode run over the pool
    quantised once beforehand (untimed).
    Returns GB/s over the sample's algorithmic bytes.
    """
    import numpy as np

    from oracle import attention as OA
    from oracle import cache as OC
    from oracle.allocator import BlockAllocatorModel
    from paged_kv_cache_283_gb300 import inputs as I

    w = I.workload(idx)
    m = BlockAllocatorModel(w.num_blocks, w.block_size, w.free_order)
    for b, n in enumerate(w.context_lens.tolist()):
        m.add_seq(b)
        m.reserve(b, n - 1)
    slots = np.array([x[0] for x in m.append_slots(range(w.num_seqs))], dtype=np.int64)
    tables = [m.block_table(b) for b in range(w.num_seqs)]

    def run(nseq):
        OC.reshape_and_cache(w.key[:nseq], w.value[:nseq], w.k_cache, w.v_cache, slots[:nseq],
                             w.block_size, inplace=True)
        for b in range(nseq):
            OA.decode_sequence(w.q[b], w.k_cache, w.v_cache, tables[b], int(w.context_lens[b]),
                               w.scale, w.block_size)

    if kv == "int8":
        from oracle import quant as OQ
        kc8, ks8 = OQ.quantize_int8(w.k_cache)
        vc8, vs8 = OQ.quantize_int8(w.v_cache)

        def run(nseq):  # noqa: F811
            OQ.reshape_and_cache_int8(w.key[:nseq], w.value[:nseq], kc8, vc8, ks8, vs8,
                                      slots[:nseq], w.block_size, inplace=True)
            OQ.decode_int8(w.q[:nseq], kc8, vc8, ks8, vs8, tables[:nseq],
                           w.context_lens[:nseq], w.scale, w.block_size)
    elif kv == "fp8":
        from oracle import fp8 as OF
        kc8, ks8 = OF.quantize_fp8(w.k_cache)
        vc8, vs8 = OF.quantize_fp8(w.v_cache)

        def run(nseq):  # noqa: F811
            OF.reshape_and_cache_fp8(w.key[:nseq], w.value[:nseq], kc8, vc8, ks8, vs8,
                                     slots[:nseq], w.block_size, inplace=True)
            OF.decode_fp8(w.q[:nseq], kc8, vc8, ks8, vs8, tables[:nseq],
                          w.context_lens[:nseq], w.scale, w.block_size)

    nseq = 1
    while True:
        t = time.perf_counter()
        run(nseq)
        dt = time.perf_counter() - t
        if dt >= 0.2 or nseq >= w.num_seqs:
            break
        nseq = min(w.num_seqs, nseq * 2)
    reps, total = 0, 0.0
    while total < max_seconds or reps == 0:
        t = time.perf_counter()
        run(nseq)
        total += time.perf_counter() - t
        reps += 1
    nbytes = decode_bytes(w.context_lens[:nseq], nseq, w.num_q_heads, w.num_kv_heads,
                          w.head_dim, w.block_size, kv) + cache_write_bytes(
                              nseq, w.num_kv_heads, w.head_dim, kv)
    threads = os.environ.get("OMP_NUM_THREADS", "")
    cores = int(threads) if threads.isdigit() else os.cpu_count()
    res = {"value": nbytes * reps / total / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
           "blas_threads": cores, "host_cpus": os.cpu_count(),
           "sample": f"first {nseq} of {w.num_seqs} sequences of the step (cache write + "
                     f"float64 decode, {kv} KV), {reps} repetitions, {total:.1f} s",
           "seconds_per_sample": total / reps, "seqs": nseq, "bytes_per_sample": nbytes}
    if out_json:
        print(json.dumps(res))
    return res


def _oracle_process(idx, seconds, kv, threads):
    """oracle_step_sample in a fresh process without CUDA, its BLAS (and
    OpenMP) thread count set to ``threads``."""
    t = str(threads)
    env = dict(os.environ, OMP_NUM_THREADS=t, OPENBLAS_NUM_THREADS=t, MKL_NUM_THREADS=t,
               CUDA_VISIBLE_DEVICES="")
    code = ("import bench, sys; bench.oracle_step_sample(%d, %f, kv=%r)" % (idx, seconds, kv))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    if r.returncode != 0:
        return {"value": None, "unit": UNIT, "cores": threads, "kind": "oracle",
                "sample": "failed: " + r.stderr.strip().splitlines()[-1][:200]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(idx, seconds, kv="bf16"):
    """The float64 oracle on the host: once with every host CPU available to
    its BLAS (the reported baseline) and once on one thread (``one_core``)."""
    ncpu = os.cpu_count() or 1
    res = _oracle_process(idx, seconds, kv, ncpu)
    res["one_core"] = _oracle_process(idx, seconds, kv, 1)
    return res


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    if os.environ.get("OMP_NUM_THREADS") != "1":
        # time the oracle on exactly one host thread, in a fresh process
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1",
                   MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
        env.pop("RANK", None)
        env.pop("WORLD_SIZE", None)
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--gpus", str(args.gpus), "--steps", str(args.steps),
                            "--warmup", str(args.warmup), "--workload", str(args.workload)],
                           env=env, cwd=ROOT)
        return r.returncode
    # one oracle sample per step, sized so that warmup + steps stay within ~2 minutes
    probe = oracle_step_sample(args.workload, 0.0, out_json=False)
    per = probe["seconds_per_sample"]
    budget = 120.0 / max(1, args.steps + args.warmup)
    import math
    from paged_kv_cache_283_gb300 import inputs as I
    w = I.workload(args.workload, with_data=False)
    nseq = max(1, min(probe["seqs"], int(math.floor(probe["seqs"] * budget / per))))
    res = _reference_timed(args, nseq)
    print(json.dumps(res))
    return 0


def _reference_timed(args, nseq):
    import numpy as np

    from oracle import attention as OA
    from oracle import cache as OC
    from oracle.allocator import BlockAllocatorModel
    from paged_kv_cache_283_gb300 import inputs as I

    w = I.workload(args.workload)
    m = BlockAllocatorModel(w.num_blocks, w.block_size, w.free_order)
    for b, n in enumerate(w.context_lens.tolist()):
        m.add_seq(b)
        m.reserve(b, n - 1)
    slots = np.array([x[0] for x in m.append_slots(range(w.num_seqs))], dtype=np.int64)
    tables = [m.block_table(b) for b in range(w.num_seqs)]

    def step():
        OC.reshape_and_cache(w.key[:nseq], w.value[:nseq], w.k_cache, w.v_cache, slots[:nseq],
                             w.block_size, inplace=True)
        for b in range(nseq):
            OA.decode_sequence(w.q[b], w.k_cache, w.v_cache, tables[b], int(w.context_lens[b]),
                               w.scale, w.block_size)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    nbytes = decode_bytes(w.context_lens[:nseq], nseq, w.num_q_heads, w.num_kv_heads,
                          w.head_dim, w.block_size) + cache_write_bytes(nseq, w.num_kv_heads,
                                                                        w.head_dim)
    value = nbytes * args.steps / dt / 1e9
    threads = os.environ.get("OMP_NUM_THREADS") or str(os.cpu_count())
    # the GPU arm's workload keys; the oracle runs one layer of it on the host
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.num_seqs, "layers": 1,
                       "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
                       "head_dim": w.head_dim, "block_size": w.block_size,
                       "num_blocks": w.num_blocks,
                       "mean_context": float(np.mean(w.context_lens)),
                       "new_tokens_per_step": w.num_seqs, "kv_cache": "bf16",
                       "attention": "float64 oracle on one host thread: "
                                    "oracle.cache.reshape_and_cache + "
                                    "oracle.attention.decode_sequence per sequence",
                       "sample_seqs": nseq,
                       "parallelism": "rank 0 only, host cores (no GPU)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle",
                             "cores": int(threads) if threads.isdigit() else threads,
                             "sample": f"first {nseq} of {w.num_seqs} sequences per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------
# multi-rank aggregation (weak scaling: every rank times its own batch)

def combine_ranks(local_seconds, step_bytes, steps, world, device="cpu"):
    """Max of the ranks' timed seconds and the whole-job GB/s it implies.

    Each rank processed ``steps`` steps of ``step_bytes`` algorithmic bytes;
    the job took as long as the slowest rank.  Host-side timing exchange only:
    the data path has no collective.
    """
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(local_seconds)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dt = float(t.item())
    return dt, world * step_bytes * steps / dt / 1e9


# ---------------------------------------------------------------------------
# GPU arm

def _setup(idx, device, replicas_min_bytes, kv_dtype="bf16", max_layers=None, n_replicas=None):
    """Device inputs of a workload: block tables and slots from the library's
    allocator, pool replicas (each larger than L2, or one pool per layer),
    q and the new tokens' K/V.  max_layers (tests, profiling) builds only the
    first layers of the 32-layer workload (each layer's launch is the same);
    n_replicas (profiling) sets the number of pool replicas of a one-layer
    workload (default: enough to exceed replicas_min_bytes, at least 2)."""
    import numpy as np
    import torch

    from paged_kv_cache_283_gb300 import inputs as I
    from paged_kv_cache_283_gb300 import pa

    w = I.workload(idx)
    alloc = pa.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    seqs = list(range(w.num_seqs))
    if idx == 4:
        alloc.add_seq(-1)
        alloc.reserve(-1, w.prefix_len)
        for b, s in enumerate(w.suffix_lens.tolist()):
            alloc.fork(-1, b)
            alloc.reserve(b, s - 1)
        alloc.free_seq(-1)
    else:
        for b, n in enumerate(w.context_lens.tolist()):
            alloc.add_seq(b)
            alloc.reserve(b, n - 1)
    slots, cow_src, _ = alloc.append_slots(seqs)
    assert np.all(cow_src == -1)
    bt, ctx = alloc.block_tables(seqs, w.max_blocks_per_seq)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(
            torch.bfloat16)

    pool_bytes = 2 * w.k_cache.nbytes
    layers = w.layers if max_layers is None else min(w.layers, max_layers)
    if layers > 1:
        # one pool per layer, each a seeded block permutation of the base pool
        base_k, base_v = bf(w.k_cache), bf(w.v_cache)
        pools = []
        for layer in range(layers):
            order = torch.from_numpy(I.layer_block_order(w, layer)).to(device)
            pools.append((base_k.index_select(0, order), base_v.index_select(0, order)))
        del base_k, base_v
        per_layer = [I.layer_inputs(w, layer) for layer in range(layers)]
        qs = [bf(x[0]) for x in per_layer]
        keys = [bf(x[1]) for x in per_layer]
        vals = [bf(x[2]) for x in per_layer]
        replicas = [pools]
    else:
        nrep = n_replicas or max(2, -(-replicas_min_bytes // pool_bytes))
        k0, v0 = bf(w.k_cache), bf(w.v_cache)
        replicas = [[(k0, v0)]] + [[(k0.clone(), v0.clone())] for _ in range(nrep - 1)]
        qs, keys, vals = [bf(w.q)], [bf(w.key)], [bf(w.value)]
    if kv_dtype in ("int8", "fp8"):
        # synthetic 1-byte pools of the same shape: INT8 codes uniform in
        # [-127, 127], scales as N(0, 1) rows give (about 3.5 / 127); FP8 codes
        # uniform over the finite E4M3 codes (never 0x7F / 0xFF), scales about
        # 3.5 / 448
        gen = torch.Generator(device=device)
        gen.manual_seed(283 + idx)

        def codes(shape):
            if kv_dtype == "int8":
                return torch.randint(-127, 128, shape, generator=gen, device=device,
                                     dtype=torch.int8)
            mag = torch.randint(0, 0x7F, shape, generator=gen, device=device, dtype=torch.int32)
            sign = torch.randint(0, 2, shape, generator=gen, device=device, dtype=torch.int32)
            return (mag | (sign << 7)).to(torch.uint8)

        lo = 0.02 if kv_dtype == "int8" else 0.006

        def int8_pool():
            nb = w.num_blocks
            shape = (nb, w.num_kv_heads, w.block_size, w.head_dim)
            v = codes(shape)
            if kv_dtype == "int8":  # V bytes are stored offset binary (code + 128)
                v = torch.bitwise_xor(v, torch.tensor(-128, dtype=torch.int8, device=device))
            return (codes(shape), v,
                    torch.rand(shape[:3], generator=gen, device=device) * lo / 2 + lo,
                    torch.rand(shape[:3], generator=gen, device=device) * lo / 2 + lo)
        pool_bytes = 2 * w.num_blocks * w.num_kv_heads * w.block_size * (w.head_dim + 4)
        if layers > 1:
            replicas = [[int8_pool() for _ in range(layers)]]
        else:
            nrep = n_replicas or max(2, -(-replicas_min_bytes // pool_bytes))
            replicas = [[int8_pool()] for _ in range(nrep)]
    st = {
        "w": w, "bt": torch.from_numpy(bt).to(device), "ctx": torch.from_numpy(ctx).to(device),
        "slots": torch.from_numpy(slots).to(device), "replicas": replicas, "q": qs,
        "key": keys, "value": vals, "bt_host": bt, "ctx_host": ctx, "slots_host": slots,
        "pool_bytes": pool_bytes, "kv": kv_dtype,
    }
    return st


def _attn_fns(st, attn, partition, fused=True, order=None, early_read=False,
              shared_prefix=False):
    import torch

    from paged_kv_cache_283_gb300 import pa

    w = st["w"]
    outs = [torch.empty_like(q) for q in st["q"]]
    ws = None
    if attn == "splitk":
        ws = pa.splitk_workspace(w.num_seqs, w.num_q_heads, w.head_dim,
                                 int(w.context_lens.max()), partition, st["q"][0].device)

    if shared_prefix:
        # the shared-prefix step: the prefix's partitions for the whole batch
        # on the tensor cores, the rest by split-K with the cache write and
        # the merge (two launches per layer)
        dev = st["q"][0].device
        sp_ws = pa.shared_prefix_workspace(w.num_seqs, w.num_q_heads, w.head_dim,
                                           int(w.context_lens.max()), w.prefix_len,
                                           SHARED_PREFIX_SPLIT, partition, dev)
        sp_cnt = pa.step_counters(w.num_seqs, w.num_kv_heads, dev)
        if order is None:
            order = torch.from_numpy(pa.shared_prefix_order(
                w.context_lens, w.prefix_len, partition, sp_ws[1].shape[2],
                SHARED_PREFIX_SPLIT)).to(dev)

        def prefix_layer(layer, *pool):
            pa.pa_decode_step_shared_prefix(outs[layer], st["q"][layer], pool[0], pool[1],
                                            st["bt"], st["ctx"], w.scale, w.prefix_len,
                                            SHARED_PREFIX_SPLIT, partition, sp_ws, sp_cnt,
                                            key=st["key"][layer], value=st["value"][layer],
                                            slot_mapping=st["slots"], order=order)

        def prefix_step(r):
            for layer, pool in enumerate(st["replicas"][r]):
                prefix_layer(layer, *pool)

        return prefix_step, prefix_layer, outs

    if fused:
        # one pa_decode_step launch per layer: cache write + attention (+ merge)
        counters = (pa.step_counters(w.num_seqs, w.num_kv_heads, st["q"][0].device)
                    if attn == "splitk" else None)

        def fused_layer(layer, *pool):
            scales = {"k_scales": pool[2], "v_scales": pool[3]} if len(pool) == 4 else {}
            pa.pa_decode_step(outs[layer], st["q"][layer], pool[0], pool[1], st["bt"], st["ctx"],
                              w.scale, key=st["key"][layer], value=st["value"][layer],
                              slot_mapping=st["slots"],
                              partition_size=partition if attn == "splitk" else 0,
                              workspace=ws, counters=counters, order=order,
                              early_read=early_read, **scales)

        def fused_step(r):
            for layer, pool in enumerate(st["replicas"][r]):
                fused_layer(layer, *pool)

        return fused_step, fused_layer, outs

    sfx = KV_SUFFIX[st.get("kv", "bf16")]
    f_split = getattr(pa, "pa_decode_splitk" + sfx)
    f_whole = getattr(pa, "pa_decode" + sfx)
    f_write = getattr(pa, "pa_reshape_and_cache" + sfx)

    def dominant(layer, *pool):
        q = st["q"][layer]
        if attn == "splitk":
            f_split(*ws, q, *pool, st["bt"], st["ctx"], w.scale, partition_size=partition)
        else:
            f_whole(outs[layer], q, *pool, st["bt"], st["ctx"], w.scale)

    def attend(layer, *pool):
        dominant(layer, *pool)
        if attn == "splitk":
            pa.pa_splitk_reduce(outs[layer], *ws, st["ctx"], partition_size=partition)

    def step(r):
        for layer, pool in enumerate(st["replicas"][r]):
            f_write(st["key"][layer], st["value"][layer], *pool, st["slots"])
            attend(layer, *pool)

    return step, dominant, outs


def step_launch(workload_idx, w, kv="bf16", step="fused", attn="auto", partition=None,
                order="longest", early_read="on", num_sms=None):
    """The launch arguments this benchmark times for a workload: attention
    kind, fused or separate launches, partition size (and how it was chosen),
    the host work order (numpy int32, or None for grid order) and whether the
    fused launches read early.  The GPU parity tests run the same arguments.

    * split-K for every workload (the shared-prefix batch too: one partition
      per sequence there, 98 us vs 110 us whole-sequence);
    * the partition size from pa_splitk_partition_size, except the
      long-context workload, whose configuration fixes 512-token partitions;
    * longest-first order when the fused step merges inside the launch
      (plan_decode_step);
    * early reads for fused launches: in this step sequence the kernel before
      each launch is the previous layer's or step's, which writes only its own
      pool (another replica or layer), so tables, lengths, order and this
      launch's pool are not written by it (PA_STEP_EARLY_READ's contract)."""
    from paged_kv_cache_283_gb300 import pa
    attn = "splitk" if attn == "auto" else attn
    if step == "shared-prefix":
        if not w.prefix_len or kv != "bf16":
            raise ValueError("--step shared-prefix: the shared-prefix workload, bf16 cache")
        part = partition or SHARED_PREFIX_PARTITION
        maxp = pa.shared_prefix_partitions(int(w.context_lens.max()), w.prefix_len,
                                           SHARED_PREFIX_SPLIT, part)
        return {"attn": "splitk", "fused": False, "shared_prefix": True, "partition": part,
                "partition_choice": "given" if partition else
                "%d after the prefix (the prefix: %d tensor-core partitions of %d)"
                % (part, w.prefix_len // SHARED_PREFIX_SPLIT, SHARED_PREFIX_SPLIT),
                "order": pa.shared_prefix_order(w.context_lens, w.prefix_len, part, maxp,
                                                SHARED_PREFIX_SPLIT),
                "plan": None, "early_read": False}
    fused = step == "fused"
    choice = "given"
    if partition is None and workload_idx == 3:
        partition, choice = 512, "fixed by the workload"
    plan = None
    if attn == "splitk":
        plan = pa.plan_decode_step(w.context_lens, w.num_q_heads, w.num_kv_heads, w.head_dim, kv,
                                   num_sms, partition_size=partition,
                                   order="longest" if fused and order == "longest" else "grid")
        if plan.chosen:
            choice = "pa_splitk_partition_size (makespan model)"
        partition = plan.partition_size
    return {"attn": attn, "fused": fused, "shared_prefix": False, "partition": partition,
            "partition_choice": choice, "order": plan.order if plan is not None else None,
            "plan": plan, "early_read": fused and early_read == "on"}


def recorded_traffic(kernel, workload_name, partition, sources=("decode.cu", "decode_tile.cuh")):
    """DRAM bytes per launch from the committed ncu summaries, or None when the
    kernel source (the files ``sources``) or the launch shape changed since the
    counters were taken.  ``profiles/decode_traffic.txt`` holds one
    ``key=value`` record per kernel, records separated by blank lines."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    try:
        with open(path) as f:
            blocks = f.read().split("\n\n")
        h = hashlib.sha256()
        for name in sources:
            with open(os.path.join(ROOT, "paged_kv_cache_283_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        sha = h.hexdigest()
    except OSError:
        return None
    for block in blocks:
        kv = dict(line.strip().split("=", 1) for line in block.splitlines()
                  if "=" in line and not line.startswith("#"))
        if (kv and sha.startswith(kv.get("kernel_source_sha256_prefix", "-"))
                and kv.get("kernel") == kernel and kv.get("workload") == workload_name
                and ("splitk" not in kernel or int(kv.get("partition", -1)) == partition)):
            return int(kv["dram_bytes_per_launch"])
    return None


def _capture(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def _time_graphs(graphs, count, stream):
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for k in range(count):
            graphs[k % len(graphs)].replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from paged_kv_cache_283_gb300 import pa

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"bench: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(args.workload, args.cpu_seconds, args.kv)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)  # before the process group, so NCCL binds this GPU
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    from paged_kv_cache_283_gb300 import build as _b
    _b.build()
    pa.lib()
    pa.pa_clear_device_error()
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    st = _setup(args.workload, device, 4 * l2, args.kv, max_layers=args.max_layers,
                n_replicas=args.replicas)
    w = st["w"]
    nl = len(st["replicas"][0])  # layers built (all, unless --max-layers)
    stream = torch.cuda.Stream(device)
    lp = step_launch(args.workload, w, args.kv, step=args.step, attn=args.attn,
                     partition=args.partition, order=args.order, early_read=args.early_read,
                     num_sms=torch.cuda.get_device_properties(device).multi_processor_count)
    attn, fused, early = lp["attn"], lp["fused"], lp["early_read"]
    args.partition, partition_choice = lp["partition"], lp["partition_choice"]
    ordered = lp["order"] is not None
    order = torch.from_numpy(lp["order"]).to(device) if ordered else None
    step, dominant, outs = _attn_fns(st, attn, args.partition, fused, order, early,
                                     lp["shared_prefix"])

    # eager warmup (sets kernel attributes, checks the error word)
    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            step(k % len(st["replicas"]))
    stream.synchronize()
    assert pa.pa_get_device_error() == 0, "device error word set during warmup"

    graphs = [_capture(lambda r=r: step(r), stream) for r in range(len(st["replicas"]))]
    launches_per_step = nl * (2 if lp["shared_prefix"] else
                              1 if fused else (2 if attn == "decode" else 3))

    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    sampler.start()
    # soak under the same load right before the timed steps, so that the
    # clock samples (every 200 ms) describe the clocks the steps ran at
    time.sleep(0.3)
    t_soak = time.time()
    soak = 0.0
    while soak < args.soak_seconds:
        soak += _time_graphs(graphs, 200, stream)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    dt = _time_graphs(graphs, args.steps, stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    sampler.stop()
    clocks = sampler.summary(t_soak, t1 + 0.05)
    if clocks.get("window") == "timed region":
        clocks["window"] = "%.2f s of soak under the same load + the timed steps" % soak

    # dominant kernel alone: graphs of back-to-back launches over the replicas
    def dom_all(r):
        for layer, pool in enumerate(st["replicas"][r]):
            dominant(layer, *pool)
    dom_graphs = [_capture(lambda r=r: dom_all(r), stream) for r in range(len(st["replicas"]))]
    _time_graphs(dom_graphs, 20, stream)
    n_dom = max(args.steps, 50)
    dom_dt = _time_graphs(dom_graphs, n_dom, stream) / (n_dom * nl)

    # end to end through the public API with pinned host buffers
    e2e = (_e2e(st, attn, args, stream, order, early, lp["shared_prefix"]) if not args.no_e2e
           else None)
    assert pa.pa_get_device_error() == 0, "device error word set during the run"

    step_bytes = nl * (decode_bytes(w.context_lens, w.num_seqs, w.num_q_heads,
                                          w.num_kv_heads, w.head_dim, w.block_size, args.kv)
                             + cache_write_bytes(w.num_seqs, w.num_kv_heads, w.head_dim,
                                                 args.kv))
    dom_bytes = decode_bytes(w.context_lens, w.num_seqs, w.num_q_heads, w.num_kv_heads,
                             w.head_dim, w.block_size, args.kv)
    if fused:  # the fused kernel also does the cache write
        dom_bytes += cache_write_bytes(w.num_seqs, w.num_kv_heads, w.head_dim, args.kv)
    dt_max, value = combine_ranks(dt, step_bytes, args.steps, world, device)
    hbm_peak = peaks.get("hbm_gbs")
    achieved = dom_bytes / dom_dt / 1e9
    if lp["shared_prefix"]:
        kname = kkey = "pa_decode_step_shared_prefix (prefix partials; split-K rest + merge)"
    elif fused:
        kname = ("pa_decode_step" + KV_SUFFIX[args.kv]
                 + (" (split-K %d, merged in-kernel)" % args.partition if attn == "splitk"
                    else " (whole sequence)"))
        kkey = "pa_decode_step" + KV_SUFFIX[args.kv] + ("_splitk" if attn == "splitk" else "")
    else:
        kname = kkey = ("pa_decode_splitk" if attn == "splitk" else "pa_decode") + KV_SUFFIX[
            args.kv]
    roofline = {"bound": "hbm", "achieved": round(achieved, 1),
                "peak": hbm_peak if hbm_peak else 6800.0, "unit": "GB/s",
                "frac": round(achieved / (hbm_peak if hbm_peak else 6800.0), 4),
                "traffic": args.traffic if args.traffic is not None else recorded_traffic(
                    kkey, w.name, args.partition,
                    ("decode.cu", "decode_tile.cuh", "prefill.cu") if lp["shared_prefix"]
                    else ("decode.cu", "decode_tile.cuh")),
                "kernel": kname,
                "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if hbm_peak
                else "fallback 6.8 TB/s",
                "bytes_per_launch": dom_bytes, "us_per_launch": round(dom_dt * 1e6, 2)}
    sfx = KV_SUFFIX[args.kv]
    if lp["shared_prefix"]:
        attention = ("pa_decode_step_shared_prefix: the %d-token prefix as %d tensor-core "
                     "partitions for the whole batch, the rest by split-K (partition %d) with "
                     "the cache write and the merge (two launches)"
                     % (w.prefix_len, w.prefix_len // SHARED_PREFIX_SPLIT, args.partition))
    elif fused:
        attention = ("pa_decode_step%s: cache write + split-K (partition %d) + merge in one launch"
                     % (sfx, args.partition) if attn == "splitk" else
                     "pa_decode_step%s: cache write + whole-sequence decode in one launch" % sfx)
    else:
        attention = ("pa_reshape_and_cache%s, pa_decode_splitk%s, pa_splitk_reduce, partition %d"
                     % (sfx, sfx, args.partition) if attn == "splitk" else
                     "pa_reshape_and_cache%s, pa_decode%s" % (sfx, sfx))
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt_max / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.kv, "data": "synthetic",
        "config": {
            "workload": w.name, "batch": w.num_seqs, "layers": nl,
            "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "num_blocks": w.num_blocks,
            "mean_context": float(np.mean(w.context_lens)), "new_tokens_per_step": w.num_seqs,
            "attention": attention,
            "kv_cache": args.kv,
            "graph": "one CUDA graph per step (cache write + attention)",
            "step": args.step,
            "early_read": early,
            "partition": args.partition if attn == "splitk" else None,
            "partition_choice": partition_choice if attn == "splitk" else None,
            "work_order": ("longest first (pa_splitk_order)" if ordered else "grid")
            if attn == "splitk" else None,
            "l2": "pool rotated over %d replicas of %.0f MB (> L2 %.0f MB)"
                  % (len(st["replicas"]), st["pool_bytes"] / 1e6, l2 / 1e6)
            if len(st["replicas"]) > 1 else "32 distinct per-layer pools per step",
            "parallelism": "dp%d (independent sequences per GPU)" % world,
        },
        "seq_layers_per_s": round(world * w.num_seqs * nl * args.steps / dt_max, 1),
        "tokens_per_s": round(world * w.num_seqs * args.steps / dt_max, 1),
        "frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "frac_of_measured_hbm": round(value / world / hbm_peak, 4) if hbm_peak else None,
        "bytes_per_step": step_bytes,
        "roofline": roofline,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
    }
    if w.prefix_len:
        # shared prefix: the same time over unique bytes (the prefix once)
        ub = unique_decode_bytes(w, args.kv)
        if fused:
            ub += cache_write_bytes(w.num_seqs, w.num_kv_heads, w.head_dim, args.kv)
        step_unique = nl * (unique_decode_bytes(w, args.kv) + cache_write_bytes(
            w.num_seqs, w.num_kv_heads, w.head_dim, args.kv))
        res["unique_bytes_per_step"] = step_unique
        res["value_unique"] = round(world * step_unique * args.steps / dt_max / 1e9, 1)
        roofline["achieved_unique"] = round(ub / dom_dt / 1e9, 1)
        roofline["frac_unique"] = round(ub / dom_dt / 1e9 / roofline["peak"], 4)
        roofline["bytes_per_launch_unique"] = ub
    if base is not None:
        res["cpu_baseline"] = base
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        dist.destroy_process_group()
    return 0


def _e2e(st, attn, args, stream, order=None, early=False, shared_prefix=False):
    """Same metric through the public API: every step, the step's inputs (q,
    the new tokens' K/V, slots, block tables, context lengths, all layers)
    go from a pinned host buffer to the device in one copy, the library's step
    objects run, and the output comes back to pinned host memory; wall clock
    around all steps.  As in a serving loop, two buffer sets alternate: step
    k + 1's inputs are copied in (one copy stream) and step k's output out
    (another) while step k computes, with events ordering every reuse."""
    import torch

    from paged_kv_cache_283_gb300 import pa

    w = st["w"]
    dev = st["bt"].device
    layers = len(st["replicas"][0])
    pieces = []
    for layer in range(layers):
        pieces += [("q", layer, st["q"][layer]), ("key", layer, st["key"][layer]),
                   ("value", layer, st["value"][layer])]
    pieces += [("slots", 0, st["slots"]), ("bt", 0, st["bt"]), ("ctx", 0, st["ctx"])]
    if order is not None:  # the step's work order is one of its inputs
        pieces.append(("order", 0, order))
    offs, total = [], 0
    for _, _, t in pieces:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    nrep = len(st["replicas"])
    ws = None
    if attn == "splitk":
        ws = pa.splitk_workspace(w.num_seqs, w.num_q_heads, w.head_dim,
                                 int(w.context_lens.max()), args.partition, dev)
    sets = []
    for s in range(2):
        host = torch.empty(total, dtype=torch.uint8).pin_memory()
        staged = torch.empty(total, dtype=torch.uint8, device=dev)
        views = {}
        for (name, layer, t), off in zip(pieces, offs):
            n = t.numel() * t.element_size()
            host[off:off + n].copy_(t.contiguous().view(torch.uint8).reshape(-1).cpu())
            views[(name, layer)] = staged[off:off + n].view(t.dtype).view(t.shape)
        out = torch.empty((layers,) + tuple(st["q"][0].shape), dtype=torch.bfloat16, device=dev)
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        def sp_step(l, pool, views=views, out=out):
            sp_ws = pa.shared_prefix_workspace(w.num_seqs, w.num_q_heads, w.head_dim,
                                               int(w.context_lens.max()), w.prefix_len,
                                               SHARED_PREFIX_SPLIT, args.partition, dev)
            sp_cnt = pa.step_counters(w.num_seqs, w.num_kv_heads, dev)
            return pa.SharedPrefixStep(
                out[l], views[("q", l)], pool[0], pool[1], views[("bt", 0)], views[("ctx", 0)],
                w.scale, w.prefix_len, SHARED_PREFIX_SPLIT, args.partition, sp_ws, sp_cnt,
                key=views[("key", l)], value=views[("value", l)], slot_mapping=views[("slots", 0)],
                order=views[("order", 0)] if order is not None else None, stream=stream)
        if shared_prefix:
            sets.append({"host": host, "staged": staged, "out": out, "hout": hout,
                         "steps": [[sp_step(l, pool) for l, pool in enumerate(st["replicas"][r])]
                                   for r in range(nrep)],
                         "in_done": torch.cuda.Event(), "computed": torch.cuda.Event(),
                         "out_done": torch.cuda.Event()})
            continue
        steps = [[pa.DecodeStep(views[("key", l)], views[("value", l)], pool[0], pool[1],
                                views[("slots", 0)], views[("q", l)], views[("bt", 0)],
                                views[("ctx", 0)], out[l], w.scale, split=attn == "splitk",
                                partition_size=args.partition, workspace=ws, stream=stream,
                                k_scales=pool[2] if len(pool) == 4 else None,
                                v_scales=pool[3] if len(pool) == 4 else None,
                                fused=args.step == "fused",
                                order=views[("order", 0)] if order is not None else None,
                                early_read=early)
                  for l, pool in enumerate(st["replicas"][r])] for r in range(nrep)]
        sets.append({"host": host, "staged": staged, "out": out, "hout": hout, "steps": steps,
                     "in_done": torch.cuda.Event(), "computed": torch.cuda.Event(),
                     "out_done": torch.cuda.Event()})
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)

    def one(k):
        b = sets[k % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(b["computed"])        # step k-2 has finished reading this set
            b["staged"].copy_(b["host"], non_blocking=True)
            b["in_done"].record(s_in)
        stream.wait_event(b["in_done"])
        stream.wait_event(b["out_done"])          # step k-2's output has been copied out
        for fn in b["steps"][k % nrep]:
            fn()
        b["computed"].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(b["computed"])
            b["hout"].copy_(b["out"], non_blocking=True)
            b["out_done"].record(s_out)

    for k in range(4):
        one(k)
    torch.cuda.synchronize()
    # at least E2E_MIN_SECONDS of steps (whatever --steps is), so that a short
    # run still measures the loop in its steady state
    t = time.perf_counter()
    for k in range(20):
        one(k)
    torch.cuda.synchronize()
    per = (time.perf_counter() - t) / 20
    n = max(args.steps, int(E2E_MIN_SECONDS / max(per, 1e-7)) + 1)
    t = time.perf_counter()
    for k in range(n):
        one(k)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t
    step_bytes = layers * (decode_bytes(w.context_lens, w.num_seqs, w.num_q_heads,
                                          w.num_kv_heads, w.head_dim, w.block_size, st["kv"])
                             + cache_write_bytes(w.num_seqs, w.num_kv_heads, w.head_dim,
                                                 st["kv"]))
    h2d = sum(t.numel() * t.element_size() for _, _, t in pieces)
    return {"value": round(step_bytes * n / dt / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(sets[0]["hout"].numel() * 2),
            "ms_per_step": dt / n * 1e3, "steps": n, "seconds": round(dt, 3),
            "how": ("pa.SharedPrefixStep per layer (pre-marshalled C calls; two launches); "
                    "every step one pinned " if shared_prefix else
                    "pa.DecodeStep per layer (pre-marshalled C calls; %s); every step one pinned "
                    % ("one pa_decode_step launch" if args.step == "fused"
                       else "separate cache-write / attention / merge launches")) +
                   "host->device copy of all inputs and one device->host copy of the output, "
                   "double-buffered on two copy streams; wall clock around all steps"}


def run_copy_blocks(args):
    """Copy-on-write block copies of a parallel-sampling step: 64 prompts
    forked into 4 samples each, whose shared, partly filled last blocks are
    copied in all 32 layers (256 pairs x 32 layers x K and V)."""
    import numpy as np
    import torch

    from paged_kv_cache_283_gb300 import build as _b
    from paged_kv_cache_283_gb300 import pa

    _b.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    layers, hkv, bs, d, pairs_n = 32, 8, 16, 128, 256
    nb = 2 * pairs_n + 64
    rng = np.random.default_rng(283 + 6)
    perm = rng.permutation(nb)
    pairs = torch.from_numpy(perm[:2 * pairs_n].reshape(pairs_n, 2).astype(np.int64)).to(dev)
    reps = 2
    pools = [([torch.randn(nb, hkv, bs, d, device=dev).to(torch.bfloat16) for _ in range(layers)],
              [torch.randn(nb, hkv, bs, d, device=dev).to(torch.bfloat16) for _ in range(layers)])
             for _ in range(reps)]
    stream = torch.cuda.Stream(dev)
    graphs = []
    with torch.cuda.stream(stream):
        for r in range(reps):
            pa.pa_copy_blocks(pools[r][0], pools[r][1], pairs)
    stream.synchronize()
    for r in range(reps):
        graphs.append(_capture(lambda r=r: pa.pa_copy_blocks(pools[r][0], pools[r][1], pairs),
                               stream))
    _time_graphs(graphs, args.warmup, stream)
    dt = _time_graphs(graphs, args.steps, stream) / args.steps
    nbytes = 2 * pairs_n * layers * 2 * hkv * bs * d * 2   # read + write, K and V
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    gbs = nbytes / dt / 1e9
    print(json.dumps({"metric": "copy-on-write block copy GB/s", "value": round(gbs, 1),
                      "unit": "GB/s", "us_per_call": round(dt * 1e6, 2), "bytes": nbytes,
                      "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4)
                      if peaks.get("hbm_gbs") else None,
                      "config": {"pairs": pairs_n, "layers": layers, "block_bytes": hkv * bs * d * 2,
                                 "l2": "2 pool replicas of %.0f MB" % (2 * layers * nb * hkv * bs * d * 2 / 1e6)}}))
    return 0


def prefill_flops(context_lens, query_lens, num_q_heads, head_dim):
    """Algorithmic FLOPs of causal chunked-prefill attention: the query at
    position p takes 2·(p+1)·D for QK and as many for PV, per query head."""
    import numpy as np
    total = 0
    for ctx, n in zip(np.asarray(context_lens).tolist(), np.asarray(query_lens).tolist()):
        first = ctx - n + 1                       # keys seen by the chunk's first query
        total += (first + ctx) * n // 2            # sum of (p + 1) over the chunk
    return 4 * total * num_q_heads * head_dim


def oracle_prefill_sample(max_seconds, out_json=True):
    """Times the float64 prefill oracle on a bounded sample of the chunked-
    prefill step: the last m query rows of its first sequence, m doubled until
    one sample takes >= 0.2 s; repeated until ``max_seconds``.  FLOP/s."""
    import numpy as np

    from oracle import prefill as OP
    from paged_kv_cache_283_gb300 import inputs as I

    w = I.chunked_prefill()
    order = w.free_order
    ctx0, n0 = int(w.context_lens[0]), int(w.query_lens[0])
    table0 = order[:-(-ctx0 // w.block_size)]
    q0 = w.q[:n0]

    def run(m):
        OP.prefill_sequence(q0[n0 - m:], w.k_cache, w.v_cache, table0, ctx0, w.scale,
                            w.block_size)

    m = 1
    while True:
        t = time.perf_counter()
        run(m)
        dt = time.perf_counter() - t
        if dt >= 0.2 or m >= n0:
            break
        m = min(n0, 2 * m)
    reps, total = 0, 0.0
    while total < max_seconds or reps == 0:
        t = time.perf_counter()
        run(m)
        total += time.perf_counter() - t
        reps += 1
    flops = prefill_flops([ctx0], [m], w.num_q_heads, w.head_dim)
    res = {"value": flops * reps / total / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
           "sample": f"last {m} of the {n0} query rows of the first chunk (float64 causal "
                     f"attention over {ctx0} cached tokens), {reps} repetitions, {total:.1f} s"}
    if out_json:
        print(json.dumps(res))
    return res


def run_prefill(args):
    """Chunked-prefill attention (pa_prefill) on the 16 x 512-token step."""
    import numpy as np
    import torch

    from paged_kv_cache_283_gb300 import build as _b
    from paged_kv_cache_283_gb300 import inputs as I
    from paged_kv_cache_283_gb300 import pa

    base = None
    if not args.no_cpu_baseline:
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1",
                   MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
        r = subprocess.run([sys.executable, "-c", "import bench; bench.oracle_prefill_sample(%f)"
                            % args.cpu_seconds], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=600)
        base = (json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else
                {"value": None, "kind": "oracle", "sample": "failed: " + r.stderr[-200:]})
    _b.build()
    pa.lib()
    pa.pa_clear_device_error()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = I.chunked_prefill(with_data=False)
    B = len(w.context_lens)
    alloc = pa.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    for b, n in enumerate(w.context_lens.tolist()):
        alloc.add_seq(b)
        alloc.reserve(b, n)
    mb = int(-(-w.context_lens.max() // w.block_size))
    bt, ctx = alloc.block_tables(list(range(B)), mb)
    assert np.array_equal(ctx, w.context_lens)
    qsl = np.concatenate([[0], np.cumsum(w.query_lens)]).astype(np.int32)
    T = int(qsl[-1])
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    pool_bytes = 2 * int(np.prod(shape)) * 2
    nrep = max(2, -(-4 * l2 // pool_bytes))
    gen = torch.Generator(device=dev)
    gen.manual_seed(283 + 6)
    pools = [(torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16),
              torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16))
             for _ in range(nrep)]
    d_bt = torch.from_numpy(bt).to(dev)
    d_ctx = torch.from_numpy(ctx.astype(np.int32)).to(dev)
    d_qsl = torch.from_numpy(qsl).to(dev)
    q = torch.randn((T, w.num_q_heads, w.head_dim), generator=gen, device=dev).to(torch.bfloat16)
    out = torch.empty_like(q)
    qmax = int(w.query_lens.max())
    stream = torch.cuda.Stream(dev)

    def call(r, qq=q, oo=out):
        pa.pa_prefill(oo, qq, pools[r][0], pools[r][1], d_bt, d_ctx, d_qsl, qmax, w.scale)

    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            call(k % nrep)
    stream.synchronize()
    assert pa.pa_get_device_error() == 0, "device error word set during warmup"
    graphs = [_capture(lambda r=r: call(r), stream) for r in range(nrep)]
    steps = max(args.steps // 10, 20)
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    # soak under the same load right before the timed steps, so that the
    # clock samples (every 20 ms) describe the clocks the steps ran at
    t_soak = time.time()
    soak = 0.0
    while soak < args.soak_seconds:
        soak += _time_graphs(graphs, 20, stream)
    t0 = time.time()
    dt = _time_graphs(graphs, steps, stream) / steps
    t1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_soak, t1 + 0.05)
    if clocks.get("window") == "timed region":
        clocks["window"] = "%.2f s of soak under the same load + the timed steps" % soak

    # end to end through the public API: q from pinned host memory in, out back
    hq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    hq.copy_(q)
    ho = torch.empty_like(hq, pin_memory=True)
    dq2, do2 = torch.empty_like(q), torch.empty_like(q)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(steps // 2, 10)
    with torch.cuda.stream(stream):
        for k in range(3 + n_e2e):
            if k == 3:
                e0.record(stream)
            dq2.copy_(hq, non_blocking=True)
            call(k % nrep, dq2, do2)
            ho.copy_(do2, non_blocking=True)
        e1.record(stream)
    stream.synchronize()
    e2e_dt = e0.elapsed_time(e1) / 1e3 / n_e2e
    assert pa.pa_get_device_error() == 0, "device error word set during the run"

    flops = prefill_flops(w.context_lens, w.query_lens, w.num_q_heads, w.head_dim)
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    tflops = flops / dt / 1e12
    peak = peaks.get("bf16_tflops")
    res = {
        "metric": "chunked-prefill attention TFLOP/s", "value": round(tflops, 2),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "tokens_per_step": T, "q_heads": w.num_q_heads,
                   "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "mean_context": float(np.mean(w.context_lens)),
                   "attention": "pa_prefill (tcgen05, one CTA per 32 tokens x 4 heads)",
                   "l2": "pool rotated over %d replicas of %.0f MB (> L2 %.0f MB)"
                         % (nrep, pool_bytes / 1e6, l2 / 1e6)},
        "flops_per_step": flops,
        "tokens_per_s": round(T / dt, 1),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 2),
                     "peak": peak if peak else 1900.0, "unit": "TFLOP/s",
                     "frac": round(tflops / (peak if peak else 1900.0), 4),
                     "traffic": recorded_traffic("pa_prefill", w.name, 0, ("prefill.cu",)),
                     "kernel": "pa_prefill",
                     "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
                     if peak else "fallback 1.9 PFLOP/s",
                     "us_per_launch": round(dt * 1e6, 2)},
        "e2e": {"value": round(flops / e2e_dt / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": q.numel() * 2, "d2h_bytes_per_step": q.numel() * 2},
        "clocks": clocks,
        "gpu_launches": steps,
    }
    if base is not None:
        res["cpu_baseline"] = base
    print(json.dumps(res))
    return 0


def main(argv=None):
    global SHARED_PREFIX_SPLIT
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=2, choices=[2, 3, 4, 5])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "int8", "fp8"],
                    help="KV cache element type (int8 / fp8 E4M3: one fp32 scale per token "
                         "and head)")
    ap.add_argument("--op", default="step", choices=["step", "copy_blocks", "prefill"],
                    help="copy_blocks: time pa_copy_blocks on a parallel-sampling step; "
                         "prefill: time pa_prefill on a 16 x 512-token chunked-prefill step")
    ap.add_argument("--attn", default="auto", choices=["auto", "decode", "splitk"],
                    help="auto (default): split-K with the chosen partition size; decode: one "
                         "CTA per (sequence, KV head)")
    ap.add_argument("--early-read", default="on", choices=["on", "off"],
                    help="fused step: read tables, lengths and pools before waiting for "
                         "the previous kernel (PA_STEP_EARLY_READ; the bench's step sequence "
                         "keeps its contract)")
    ap.add_argument("--order", default="longest", choices=["longest", "grid"],
                    help="fused split-K: CTAs handed out longest first (pa_splitk_order) "
                         "or in grid order")
    ap.add_argument("--prefix-split", type=int, default=None,
                    help="--step shared-prefix: tokens per tensor-core prefix partition "
                         "(default %d)" % SHARED_PREFIX_SPLIT)
    ap.add_argument("--step", default="fused", choices=["fused", "separate", "shared-prefix"],
                    help="fused: one pa_decode_step launch per layer (cache write + attention "
                         "+ split-K merge); separate: the cache write, partition pass and "
                         "merge as three launches; shared-prefix (the shared-prefix workload): "
                         "pa_decode_step_shared_prefix, the prefix on the tensor cores once "
                         "for the whole batch")
    ap.add_argument("--partition", type=int, default=None,
                    help="split-K partition size in tokens (default: 512 for the long-context "
                         "workload, else chosen by pa_splitk_partition_size)")
    ap.add_argument("--soak-seconds", type=float, default=0.5)
    ap.add_argument("--no-e2e", action="store_true",
                    help="profiling: skip the end-to-end leg (its thousands of launches)")
    ap.add_argument("--max-layers", type=int, default=None,
                    help="profiling: build only the first layers of the 32-layer workload "
                         "(each layer's launch is unchanged; the line then reports those layers)")
    ap.add_argument("--replicas", type=int, default=None,
                    help="profiling: pool replicas of a one-layer workload (default: enough to "
                         "exceed 4x L2, at least 2)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the dominant kernel from an ncu capture")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.prefix_split:
        SHARED_PREFIX_SPLIT = args.prefix_split
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "copy_blocks":
        return run_copy_blocks(args)
    if args.op == "prefill":
        return run_prefill(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
