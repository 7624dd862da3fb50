"""Benchmark of the quantized sparse MoE layer forward on one GB300 (or N independent replicas).

Default run (``--workload all``): the five GLM-5.2-class workloads, each on its own
resident expert set, with the decode layer at T=1 as the headline of the JSON
line and the others under ``variants``:
  decode T=1 / T=4  d=7168, d_ff=2048, 256 experts, top-8, int4 group-128, routed scale 2.5, bias 0
  mtp_verify T=3    the same plus a shared int4 expert, router bias N(0, std 0.5)
  prefill T=2048    the same plus a shared expert, Zipf-skewed router bias
  stacked T=256     six layers (int4 / int8 alternating) with RMSNorm and residual, 51.4 GB resident
A step is one full forward (router, grouping, gate/up + SwiGLU, down, combine; for the stacked workload
the whole stack; for the indexer one scoring + selection of every query token) on a fresh x, so routing differs every step; every expert set is far larger than L2.
Each entry carries its own roofline, end-to-end figure, CPU baseline (the oracle), clock record and
routing statistics (near-tie tokens, unique experts per step).

  decode + cache    decode T=1 with every expert in pinned host memory behind 32 device slots (weighted LRU)
  decode + pilot    two such layers, layer 1's experts predicted from layer 0's input and read ahead
  IDOT              decode T=1 and prefill T=2048 with integer-dot expert inputs (int8 per block of 32)
  indexer T=1 / T=4 sparse-attention key selection: 64 heads of 128, 65,536 cached keys, top-2048

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all|decode|mtp_verify|prefill|stacked|indexer]
  python bench.py --impl reference ...   # the fp64 oracle on the host cores (CPU baseline arm)

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import contextlib
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

import harness as H  # noqa: E402

METRIC = "MoE-layer tokens/s and HBM GB/s (decode) / tensor % peak (prefill) on 1 GB300"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- clocks sampling

class ClockSampler:
    """nvidia-smi SM clock / throttle-reason sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- workload

def workload_setup(name: str, experts: int = 0, tokens: int = 0):
    """(workload, T of the JSON line, all T measured).  `experts` / `tokens` shrink the workload for
    profiler captures (a few GB on the device); the default bench line uses the full configuration."""
    import dataclasses
    w = H.WORKLOADS[name]
    if experts:
        w = dataclasses.replace(w, E=experts)
    Ts = {"decode": (1, 4), "mtp_verify": (3,), "prefill": (2048,), "stacked": (256,)}[name]
    if tokens:
        Ts = (tokens,)
    return w, Ts[0], Ts


def qmat_bytes(qtype: int, N: int, K: int) -> int:
    """Packed bytes of one [N][K] expert matrix: int4-g128 codes + fp16 scales + zero-point nibbles,
    or int8 codes + fp32 scale + uint8 zero point per row."""
    if qtype == H.Q_INT4_G128:
        G = K // 128
        return N * K // 2 + N * G * 2 + N * ((G + 1) // 2)
    return N * K + N * 4 + N


def expert_set_bytes(w) -> int:
    """Bytes of all experts of every layer of workload w (routed and shared), as resident in HBM."""
    total = 0
    for qt in w.qtypes:
        per = 2 * qmat_bytes(qt, w.F, w.d) + qmat_bytes(qt, w.d, w.F)
        total += w.E * per
        if w.F_shared:
            total += 2 * qmat_bytes(qt, w.F_shared, w.d) + qmat_bytes(qt, w.d, w.F_shared)
    return total


def workload_config(w, T: int, world: int) -> dict:
    """The JSON line's `config`: the workload alone (both arms print the same one)."""
    if w.n_layers > 1:
        return {"workload": f"stacked: {w.n_layers} GLM-5.2-class MoE layers (int4, int8 alternating) with "
                            f"RMSNorm and residual, T={T} tokens per step",
                "d": w.d, "d_ff": w.F, "E": w.E, "k": w.k, "routed_scale": w.rho, "layers": w.n_layers,
                "parallelism": "replicas" if world > 1 else "single GPU",
                "l2": "inputs larger than L2: expert set of %.1f GB, fresh x every step" % (expert_set_bytes(w) / 1e9)}
    return {"workload": f"{w.name}: GLM-5.2-class MoE layer, T={T} tokens per step",
            "d": w.d, "d_ff": w.F, "E": w.E, "k": w.k, "routed_scale": w.rho,
            "qtype": "int4-g128" if w.qtypes[0] == H.Q_INT4_G128 else "int8-pc",
            "shared_expert_d_ff": w.F_shared, "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": "inputs larger than L2: expert set of %.2f GB, fresh x (fresh routing) every step"
                  % (expert_set_bytes(w) / 1e9)}


def unique_expert_bytes(dl, T, idx=None) -> tuple[int, int]:
    """(gate+up bytes, down bytes) streamed by the last forward: unique routed experts + shared."""
    if idx is None:
        idx = dl.routing(T)[0]
    U = len(np.unique(idx))
    L = dl.layer
    gu = L.experts.gate.nbytes // L.E + L.experts.up.nbytes // L.E
    dn = L.experts.down.nbytes // L.E
    gub, dnb = U * gu, U * dn
    if L.shared is not None:
        gub += L.shared.gate.nbytes + L.shared.up.nbytes
        dnb += L.shared.down.nbytes
    return gub, dnb


# DRAM bytes per launch of the dominant decode kernel, from the ncu capture summarised in
# profiles/decode_ffn_int4_T1_E32.txt (dram__bytes_read.sum + dram__bytes_write.sum of the T=1 gate/up
# launch; the launch reads the 8 selected experts, the same bytes as with E=256).  Set to None whenever
# that kernel changes, until it is captured again.
DECODE_GATEUP_T1_TRAFFIC = 122_084_096 + 3_338_240

# DRAM bytes per launch of the prefill gate/up grouped GEMM at T=2048, E=256, scaled from the capture
# summarised in profiles/prefill_ffn_int4_E64_T512.txt (T=512, E=64: 1,081,396,000 B read + 17,395,456 B
# written).  Both the expert bytes and the gathered activations grow with E and T by the same factor 4
# (the one shared expert does not: 15 MB of the 4.4 GB); the full-size launch is too large to capture
# with more than a one-pass metric.  None whenever that kernel changes.
PREFILL_GATEUP_T2048_TRAFFIC = 4 * (1_081_396_000 + 17_395_456)

# DRAM bytes per launch of the key-selection scores kernel at T=1 over 65,536 keys, from the capture
# summarised in profiles/indexer_T1_L65536.txt (the key cache read once; the scores stay in L2).
INDEXER_SCORES_T1_TRAFFIC = 16_813_312


def max_over_ranks(v: float, device=None) -> float:
    """Largest value over the ranks of the default process group (the time every replica must wait for);
    identity without one.  Replicas exchange nothing else: the layer runs independently on every GPU."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_tokens_per_s(world: int, steps: int, T: int, ms_max: float) -> float:
    """Whole-job throughput: tokens all replicas processed / the slowest replica's time."""
    return world * steps * T / (ms_max * 1e-3)


def expert_flops(layer, T: int) -> tuple[float, float]:
    """(gate/up FLOPs, down FLOPs) of one forward: every routed (token, expert) pair and every
    shared-expert row, 2 FLOPs per multiply-add; padding of the MMA N dimension is not counted."""
    pairs_f = T * layer.k * layer.F + (T * layer.F_shared if layer.shared is not None else 0)
    return 2.0 * 2 * layer.d * pairs_f, 2.0 * layer.d * pairs_f


def _timed_steps(run_step, xs, W: int, K: int, dev, world: int, stream):
    """W untimed warm-up steps, then K steps between CUDA events on the launching stream (synchronised and,
    with replicas, behind a barrier on both sides) while nvidia-smi samples the clocks.  Returns
    (device ms for the K steps, clock summary)."""
    import torch
    for i in range(W):
        run_step(xs[i])
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    with ClockSampler(dev.index) as clk:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for i in range(K):
            run_step(xs[W + i])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
    return e0.elapsed_time(e1), clk.summary()


def _e2e_steps(run_step, xs_dev, K: int, W: int, out_shape, dev):
    """The same K steps through the public API with host buffers: every step copies its x from pinned host
    memory to the device and its output back to pinned host memory inside the timed region.  Returns
    (seconds, H2D bytes per step, D2H bytes per step)."""
    import torch
    xh = [torch.empty_like(xs_dev[0], device="cpu").pin_memory() for _ in range(K)]
    for i in range(K):
        xh[i].copy_(xs_dev[W + i].cpu())
    oh = torch.empty((K,) + tuple(out_shape), dtype=torch.float32).pin_memory()
    xd = torch.empty_like(xs_dev[0])
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(K):
        xd.copy_(xh[i], non_blocking=True)
        out = run_step(xd)
        oh[i].copy_(out, non_blocking=True)
    torch.cuda.synchronize(dev)
    return time.perf_counter() - t0, xh[0].numel() * xh[0].element_size(), oh[0].numel() * 4


def bench_layer(name: str, args, dev, world: int, want_cpu: bool, cpu_budget_s: float):
    """One MoE layer workload (decode, mtp_verify or prefill): every T of the workload is timed on the same
    resident expert set.  Returns ({T: line fragment}, cpu_baseline or None, host generation seconds)."""
    import torch
    from harness.device import DeviceLayer, to_dev

    w, _, Ts = workload_setup(name, args.experts, args.tokens)
    t0 = time.time()
    layer = w.layer(0)
    dl = DeviceLayer(layer, max(Ts), device=dev)
    gen_s = time.time() - t0
    stream = torch.cuda.current_stream(dev)
    K, W = args.steps, args.warmup
    pk = peaks()
    frags = {}
    runs = [(T, False) for T in Ts]
    if name in ("decode", "prefill") and not args.experts and not args.tokens and not args.no_idot:
        runs.append((Ts[0], True))      # integer-dot expert inputs on the same layer
    for T, idot in runs:
        dl.plan.set_idot(idot)
        xs = [to_dev(w.x(T, 1000 + i), dev) for i in range(K + W)]
        out = torch.empty((T, layer.d), dtype=torch.float32, device=dev)

        def step(x):
            return dl.forward(x, out=out)

        ms, clocks = _timed_steps(step, xs, W, K, dev, world, stream)
        launches = dl.plan.last_launch_count()
        # per-kernel times: the same steps again, kernel-boundary events recorded by the library
        dl.plan.profile_begin(K)
        for i in range(K):
            step(xs[W + i])
        torch.cuda.synchronize(dev)
        kt = dl.plan.profile_end()
        # algorithmic bytes and routing statistics of these K steps (each step re-run and read back)
        gub = dnb = 0
        near = uniq = 0
        for i in range(K):
            step(xs[W + i])
            torch.cuda.synchronize(dev)
            idx, _, nt = dl.routing(T)[:3]
            a, b = unique_expert_bytes(dl, T, idx)
            gub += a
            dnb += b
            near += int(nt.sum())
            uniq += len(np.unique(idx))
        e2e_s, h2d, d2h = _e2e_steps(step, xs, K, W, (T, layer.d), dev)
        ms_tot, e2e_tot = max_over_ranks(ms, dev), max_over_ranks(e2e_s, dev)
        gu_ms, gu_n = kt.get("expert_gate_up", (0.0, 0))
        dn_ms, dn_n = kt.get("expert_down", (0.0, 0))
        layer_gbs = (gub + dnb) / K / (ms_tot / K * 1e-3) / 1e9
        if T > 8:
            # dense contraction: the tensor-core grouped GEMMs against the bf16/fp16 tensor peak
            gfl, dfl = expert_flops(layer, T)
            tg_ms, tg_n = kt.get("tc_gate_up", (0.0, 0))
            td_ms, td_n = kt.get("tc_down", (0.0, 0))
            pk_t, pk_b = pk["bf16_tflops_sustained"], pk["bf16_tflops"]
            ach = gfl / (tg_ms / tg_n * 1e-3) / 1e12 if tg_n else None
            ach_d = dfl / (td_ms / td_n * 1e-3) / 1e12 if td_n else None
            layer_tf = (gfl + dfl) / (ms_tot / K * 1e-3) / 1e12
            roof = {"bound": "tensor", "kernel": "tc_gate_up", "achieved": ach, "peak": pk_t, "unit": "TFLOP/s",
                    "frac": (ach / pk_t) if ach else None, "frac_of_burst_peak": (ach / pk_b) if ach else None,
                    "traffic": PREFILL_GATEUP_T2048_TRAFFIC if (T == 2048 and not args.experts) else None,
                    "peak_source": pk["source"] + " bf16 dense, sustained (fp16 operands run at the bf16 rate)",
                    "algorithmic_flops_per_launch": gfl, "down_kernel_achieved_tflops": ach_d,
                    "layer_tflops": layer_tf, "layer_frac_of_sustained_peak": layer_tf / pk_t,
                    "layer_frac_of_burst_peak": layer_tf / pk_b}
        else:
            achieved = (gub / gu_n) / (gu_ms / gu_n * 1e-3) / 1e9 if gu_n else None
            achieved_d = (dnb / dn_n) / (dn_ms / dn_n * 1e-3) / 1e9 if dn_n else None
            roof = {"bound": "hbm", "kernel": "expert_gate_up", "achieved": achieved, "peak": pk["hbm_gbs"],
                    "unit": "GB/s", "frac": (achieved / pk["hbm_gbs"]) if achieved else None,
                    "traffic": DECODE_GATEUP_T1_TRAFFIC if (T == 1 and name == "decode" and not args.experts)
                    else None,
                    "peak_source": pk["source"], "algorithmic_bytes_per_launch": gub / max(gu_n, 1),
                    "down_kernel_achieved_gbs": achieved_d}
        frags[(T, "idot") if idot else T] = {
            "value": replica_tokens_per_s(world, K, T, ms_tot),
            "unit": "tokens/s",
            "ms_per_step": ms_tot / K,
            "hbm_gbs_layer": layer_gbs,
            "hbm_frac_layer": layer_gbs / pk["hbm_gbs"],
            "roofline": roof,
            "kernel_ms_per_step": {k: v[0] / v[1] for k, v in kt.items()},
            "kernel_share": {k: v[0] / max(sum(x[0] for x in kt.values()), 1e-12) for k, v in kt.items()},
            "e2e": {"value": world * K * T / e2e_tot, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": K * launches,
            "clocks": clocks,
            "routing": {"tokens": K * T, "near_tie_tokens": near, "unique_experts_per_step": uniq / K,
                        "near_tie_rule": "k-th minus (k+1)-th selection score < 1e-5, flagged by the GPU router"},
            "config": dict(workload_config(w, T, world),
                           **({"activations": "integer-dot: int8 codes per block of 32, power-of-two scale"}
                              if idot else {})),
        }
        del xs
    dl.plan.set_idot(False)
    if name == "decode" and not args.experts and not args.tokens and not args.no_cache:
        frags["cache"] = bench_cache(dl, layer, w, args, dev, world)
        frags["pilot"] = bench_pilot(dl, layer, w, args, dev, world)
    # the oracle last: its threads occupy every host core, and the cache steps are driven from the host
    cpu = cpu_baseline(w, layer, Ts[0], cpu_budget_s) if want_cpu else None
    dl.close()
    del dl, layer
    torch.cuda.empty_cache()
    return frags, cpu, gen_s


def _host_tier(dl, layer):
    """Every routed expert of `layer` in one pinned host buffer, in the slot layout (each expert one
    contiguous block, so that a miss is one copy).  Returns (buffer, coli_expert per expert, slot bytes)."""
    import torch
    import quantized_expert_ffn_bias_gb300 as coli
    sb = coli.colibri_moe_cache_slot_bytes(dl.plan)
    offs = coli.cache_slot_offsets(layer.d, layer.F, layer.qtype)
    with near_gpu(dl.device):          # the pages lie in the memory of the GPU's own host
        keep = torch.empty((layer.E, sb), dtype=torch.uint8, pin_memory=True)
    kn = keep.numpy()
    for e in range(layer.E):
        for j, (n, part) in enumerate((n, p) for n in ("gate", "up", "down") for p in ("q", "s", "z")):
            src = np.ascontiguousarray(getattr(getattr(layer.experts, n), part)[e]).view(np.uint8).ravel()
            kn[e, offs[j]:offs[j] + src.size] = src
    base = keep.data_ptr()
    host = []
    for e in range(layer.E):
        b = base + e * sb
        q = [coli.qmat(b + offs[3 * m], b + offs[3 * m + 1], b + offs[3 * m + 2]) for m in range(3)]
        host.append(coli.coli_expert(q[0], q[1], q[2]))
    return keep, host, sb


def _gpu_numa(dev):
    """(NUMA node, its host cores) of the GPU's PCI device from sysfs, or None."""
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        base = f"/sys/bus/pci/devices/{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        with open(base + "/numa_node") as f:
            node = int(f.read().strip())
        if node < 0:
            return None
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            cpus = set()
            for part in f.read().strip().split(","):
                lo, _, hi = part.partition("-")
                cpus.update(range(int(lo), int(hi or lo) + 1))
        return node, cpus
    except (OSError, ValueError, AttributeError):
        return None


@contextlib.contextmanager
def near_gpu(dev):
    """Run the block on the host cores of the GPU's NUMA node, so that pinned host memory allocated in it
    lies in that node's memory (first touch) and host-to-device copies take the GPU's own host link.
    Yields the node, or None where sysfs does not name one (then nothing changes)."""
    loc = _gpu_numa(dev)
    if loc is None:
        yield None
        return
    node, cpus = loc
    old = os.sched_getaffinity(0)
    try:
        os.sched_setaffinity(0, (cpus & old) or cpus)
        yield node
    finally:
        os.sched_setaffinity(0, old)


def host_link_gbs(sb: int, dev, n: int = 8) -> float:
    """The host-to-device rate of this GPU's host link: n expert slots (sb bytes each) copied from pinned host
    memory in one copy, best of 3 (CUDA events).  The denominator of the expert-cache rooflines."""
    import torch
    with near_gpu(dev):
        src = torch.empty(n * sb, dtype=torch.uint8, pin_memory=True)
        src.fill_(1)
    dst = torch.empty(n * sb, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev)
    best = 0.0
    for _ in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        dst.copy_(src, non_blocking=True)
        e1.record(st)
        torch.cuda.synchronize(dev)
        best = max(best, n * sb / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del src, dst
    return best


def tier_copy_gbs(keep, sb: int, dev, n: int = 8) -> float:
    """The host-to-device rate out of the cache's own host tier: n experts copied in one copy, best of 3."""
    import torch
    src = keep.view(-1)[: n * sb]
    dst = torch.empty(n * sb, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev)
    best = 0.0
    for _ in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        dst.copy_(src, non_blocking=True)
        e1.record(st)
        torch.cuda.synchronize(dev)
        best = max(best, n * sb / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    return best


def bench_cache(dl, layer, w, args, dev, world: int):
    """Decode at T=1 with the experts in host memory behind a 32-slot device cache (4 x k slots, the
    walkthrough page's default), router bias Zipf-skewed (as in the prefill workload) so that experts recur.
    A step is one cached forward: routing, read-back of the chosen experts, copies of the misses from
    pinned host memory, expert kernels."""
    import torch
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import to_dev

    K, W = args.steps, args.warmup
    T, S, weight = 1, 4 * layer.k, 1.0
    bias_d = to_dev(H.gen_bias(w.seed, 0, "zipf:0.05:1.1", layer.E), dev)
    t0 = time.time()

    keep, host, sb = _host_tier(dl, layer)
    pin_s = time.time() - t0
    slots = torch.empty(S * sb, dtype=torch.uint8, device=dev)
    cache = coli.Cache(dl.plan, S, weight, host, slots, S * sb)
    stream = torch.cuda.current_stream(dev)
    xs = [to_dev(w.x(T, 5000 + i), dev) for i in range(K + W)]
    out = torch.empty((T, layer.d), dtype=torch.float32, device=dev)
    ws = torch.empty(dl.plan.workspace_bytes, dtype=torch.uint8, device=dev)

    def step(i):
        cache.forward(T, xs[i], dl.router_w, bias_d, out, ws, stream=stream)

    for i in range(W):
        step(i)
    torch.cuda.synchronize(dev)
    cache.reset_stats()
    with ClockSampler(dev.index) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(K):
            step(W + i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), dev)
    st_ = cache.stats()
    # the same routing trace through the host policy: plain LRU against the weighted rule
    sets = []
    for i in range(K + W):
        dl.plan.forward(T, xs[i], dl.router_w, bias_d, out, dl.ws, stream=stream)
        sets.append(sorted(set(dl.routing(T)[0].ravel().tolist())))

    def timed_hits(wt):
        h_all, _ = coli.colibri_moe_cache_simulate(layer.E, S, wt, sets)
        h_warm, _ = coli.colibri_moe_cache_simulate(layer.E, S, wt, sets[:W])
        return (h_all - h_warm) / max(1, sum(len(x) for x in sets[W:]))

    hit = st_["hits"] / max(1, st_["lookups"])
    copy_s = ms * 1e-3
    link = host_link_gbs(sb, dev)
    tier = tier_copy_gbs(keep, sb, dev)
    ach = st_["bytes_copied"] / copy_s / 1e9
    cache.close()
    del keep, slots
    torch.cuda.empty_cache()
    return {
        "value": replica_tokens_per_s(world, K, T, ms), "unit": "tokens/s", "ms_per_step": ms / K,
        "roofline": {"bound": "host link", "kernel": "host-to-device expert copies (misses)",
                     "achieved": ach, "peak": link, "unit": "GB/s", "frac": ach / link, "traffic": None,
                     "peak_source": "host-to-device copy of 8 expert slots from pinned memory, measured in this run "
                                    "(best of 3); achieved = bytes copied over the whole step (routing and kernels "
                                    "included)"},
        "cache": {"slots": S, "weight": weight, "hit_rate": hit, "lookups": st_["lookups"], "misses": st_["misses"],
                  "bytes_copied_per_step": st_["bytes_copied"] / K,
                  "simulated_hit_rate_plain_lru": timed_hits(0.0), "simulated_hit_rate_weighted": timed_hits(weight),
                  "host_pin_s": round(pin_s, 1), "host_numa_node": (_gpu_numa(dev) or (None,))[0],
                  "tier_copy_gbs": tier},
        "e2e": {"value": replica_tokens_per_s(world, K, T, ms), "unit": "tokens/s",
                "h2d_bytes_per_step": st_["bytes_copied"] / K, "d2h_bytes_per_step": 0},
        "gpu_launches": K * dl.plan.last_launch_count(),
        "clocks": clk.summary(),
        "config": {"workload": "decode with an expert cache: GLM-5.2-class MoE layer, T=1 tokens per step, every "
                               f"expert in pinned host memory, {S} device slots, Zipf-skewed router bias",
                   "d": layer.d, "d_ff": layer.F, "E": layer.E, "k": layer.k, "qtype": "int4-g128",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: 5.86 GB of experts in host memory, misses copied per step"},
        "cpu_baseline": None,
    }


def bench_pilot(dl0, layer0, w, args, dev, world: int):
    """Two stacked decode layers at T=1 (h <- h + MoE(bf16(RMSNorm(h))); layer 1 generated like layer 0),
    each with every expert in pinned host memory behind 32 device slots and a Zipf-skewed router bias.
    With next-layer prediction, layer 1's router runs on layer 0's normalised input on a side stream
    before layer 0, and the experts it picks are copied into layer 1's cache while layer 0 routes, copies
    and computes; layer 1 then waits for those copies.  Without it, layer 1 copies its misses after its
    own routing.  A step is both layers on a fresh input; both modes run the same inputs."""
    import torch
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import DeviceLayer, to_dev

    K, W = args.steps, args.warmup
    T, S, d, eps = 1, 4 * layer0.k, w.d, 1e-6
    t0 = time.time()
    layer1 = H.gen_layer(w.seed, 1, d=w.d, F=w.F, E=w.E, k=w.k, rho=w.rho, qtype=w.qtypes[0], bias=w.bias,
                         F_shared=w.F_shared)
    dl1 = DeviceLayer(layer1, T, device=dev)
    dls, layers = [dl0, dl1], [layer0, layer1]
    biases = [to_dev(H.gen_bias(w.seed, l, "zipf:0.05:1.1", w.E), dev) for l in range(2)]
    tiers = [_host_tier(dls[l], layers[l]) for l in range(2)]
    gen_s = time.time() - t0
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    xs = [to_dev(w.x(T, 6000 + i), dev) for i in range(K + W)]
    h, h1, h2 = (torch.empty((T, d), dtype=torch.float32, device=dev) for _ in range(3))
    n0, n1 = (torch.empty((T, d), dtype=torch.int16, device=dev) for _ in range(2))
    wss = [torch.empty(dl.plan.workspace_bytes, dtype=torch.uint8, device=dev) for dl in dls]
    wsp = torch.empty(dl1.plan.workspace_bytes, dtype=torch.uint8, device=dev)
    ev_n, ev_p = torch.cuda.Event(), torch.cuda.Event()

    def run(pilot: bool):
        sb = tiers[0][2]
        caches = [coli.Cache(dls[l].plan, S, 1.0, tiers[l][1], torch.empty(S * sb, dtype=torch.uint8, device=dev),
                             S * sb) for l in range(2)]
        preds = []

        def step(i):
            h.copy_(xs[i].view(torch.bfloat16).float())
            coli.colibri_moe_rmsnorm_bf16(h, T, d, eps, n0, stream)
            if pilot:
                ev_n.record(stream)
                side.wait_event(ev_n)
                preds.append(caches[1].pilot(T, n0, dl1.router_w, biases[1], wsp, stream=side))
                ev_p.record(side)
            caches[0].forward(T, n0, dl0.router_w, biases[0], h1, wss[0], residual=h, stream=stream)
            coli.colibri_moe_rmsnorm_bf16(h1, T, d, eps, n1, stream)
            if pilot:
                stream.wait_event(ev_p)
            caches[1].forward(T, n1, dl1.router_w, biases[1], h2, wss[1], residual=h1, stream=stream)

        for i in range(W):
            step(i)
        torch.cuda.synchronize(dev)
        for c in caches:
            c.reset_stats()
        with ClockSampler(dev.index) as clk:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(K):
                step(W + i)
            e1.record(stream)
            torch.cuda.synchronize(dev)
        ms = max_over_ranks(e0.elapsed_time(e1), dev)
        st = [c.stats() for c in caches]
        launches = dl0.plan.last_launch_count() + dl1.plan.last_launch_count() + 2
        if pilot:
            caches[1].pilot(T, n0, dl1.router_w, biases[1], wsp, stream=side)
            launches += dl1.plan.last_launch_count()
            torch.cuda.synchronize(dev)
        for c in caches:
            c.close()
        return ms, st, preds[W:], clk.summary(), launches

    ms_p, st_p, preds, clk_p, launches = run(True)
    ms_n, st_n, _, _, _ = run(False)
    # recall: layer 1's experts (resident forwards of the same steps) that the prediction named
    used = named = 0
    for i in range(K):
        h.copy_(xs[W + i].view(torch.bfloat16).float())
        coli.colibri_moe_rmsnorm_bf16(h, T, d, eps, n0, stream)
        dl0.plan.forward(T, n0, dl0.router_w, biases[0], h1, dl0.ws, dl0.ws.numel(), residual=h, stream=stream)
        coli.colibri_moe_rmsnorm_bf16(h1, T, d, eps, n1, stream)
        dl1.plan.forward(T, n1, dl1.router_w, biases[1], h2, dl1.ws, dl1.ws.numel(), stream=stream)
        torch.cuda.synchronize(dev)
        act = set(dl1.routing(T)[0].ravel().tolist())
        used += len(act)
        named += len(act & set(preds[i]))

    def hit(s):
        return s["hits"] / max(1, s["lookups"])

    copied = sum(s["bytes_copied"] for s in st_p)
    link = host_link_gbs(tiers[0][2], dev)
    ach = copied / (ms_p * 1e-3) / 1e9
    dl1.close()
    del tiers, dl1, layer1
    torch.cuda.empty_cache()
    return {
        "value": replica_tokens_per_s(world, K, T, ms_p), "unit": "tokens/s", "ms_per_step": ms_p / K,
        "roofline": {"bound": "host link", "kernel": "host-to-device expert copies (misses and read-ahead)",
                     "achieved": ach, "peak": link, "unit": "GB/s", "frac": ach / link, "traffic": None,
                     "peak_source": "host-to-device copy of 8 expert slots from pinned memory, measured in this run "
                                    "(best of 3); achieved = bytes copied over the whole step (routing and kernels "
                                    "included)"},
        "cache": {"slots_per_layer": S, "weight": 1.0,
                  "with_prediction": {"ms_per_step": ms_p / K, "hit_rate_layer0": hit(st_p[0]),
                                      "hit_rate_layer1": hit(st_p[1]),
                                      "bytes_copied_per_step": copied / K,
                                      "predicted_per_step": st_p[1]["predicted"] / K,
                                      "prefetched_per_step": st_p[1]["prefetched"] / K},
                  "without_prediction": {"ms_per_step": ms_n / K, "hit_rate_layer0": hit(st_n[0]),
                                         "hit_rate_layer1": hit(st_n[1]),
                                         "bytes_copied_per_step": sum(s["bytes_copied"] for s in st_n) / K},
                  "recall_of_layer1_experts": named / max(1, used),
                  "speedup": ms_n / ms_p,
                  "host_generation_s": round(gen_s, 1)},
        "e2e": {"value": replica_tokens_per_s(world, K, T, ms_p), "unit": "tokens/s",
                "h2d_bytes_per_step": copied / K, "d2h_bytes_per_step": 0},
        "gpu_launches": K * launches,
        "clocks": clk_p,
        "config": {"workload": "decode with expert caches and next-layer prediction: two stacked GLM-5.2-class "
                               f"MoE layers, T=1 tokens per step, every expert in pinned host memory, {S} device "
                               "slots per layer, Zipf-skewed router bias",
                   "d": w.d, "d_ff": w.F, "E": w.E, "k": w.k, "qtype": "int4-g128",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: 2 x 5.86 GB of experts in host memory, misses copied per step"},
        "cpu_baseline": None,
    }


def bench_stacked(args, dev, world: int, want_cpu: bool, cpu_budget_s: float):
    """Six stacked layers h <- h + MoE(bf16(RMSNorm(h))) per step (T=256, alternating int4 / int8 experts,
    51.4 GB resident); a step is the whole stack on a fresh input."""
    import torch
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import DeviceLayer, to_dev

    w, T, _ = workload_setup("stacked", args.experts, args.tokens)
    t0 = time.time()
    dls, expert_bytes, cpu_rates, cpu_samples = [], [], {}, []
    cores = None
    for l in range(w.n_layers):
        layer = w.layer(l)
        dl = DeviceLayer(layer, T, device=dev)
        expert_bytes.append(layer.experts.bytes_per_expert)
        if want_cpu and layer.qtype not in cpu_rates:
            # the oracle's rate on one layer of each quantisation type (the stack's cost is three of each)
            r = cpu_baseline(w, layer, T, cpu_budget_s / 2)
            cpu_rates[layer.qtype] = r["value"]
            cores = r["cores"]
            cpu_samples.append(f"layer {l} ({'int4' if layer.qtype == H.Q_INT4_G128 else 'int8'}): {r['sample']}")
        dl.experts.bank = None          # keep only the device copies
        dl.layer = None
        dls.append((dl, layer.E, layer.k))
        del layer
    gen_s = time.time() - t0
    stream = torch.cuda.current_stream(dev)
    eps = w.rmsnorm_eps
    K, W = args.steps, args.warmup
    xs = [to_dev(w.x(T, 1000 + i), dev) for i in range(K + W)]
    hb = [torch.empty((T, w.d), dtype=torch.float32, device=dev) for _ in range(2)]
    n = torch.empty((T, w.d), dtype=torch.int16, device=dev)

    def step(x, routing=None):
        h, h2 = hb
        h.copy_(x.view(torch.bfloat16).float())
        for li, (dl, E, k) in enumerate(dls):
            coli.colibri_moe_rmsnorm_bf16(h, T, w.d, eps, n, stream)
            dl.forward(n, out=h2, residual=h)
            if routing is not None:
                routing(li, dl, k)
            h, h2 = h2, h
        return h

    ms, clocks = _timed_steps(step, xs, W, K, dev, world, stream)
    ms = max_over_ranks(ms, dev)
    # per-kernel times, unique experts and near-ties per layer (the same steps again)
    for dl, _, _ in dls:
        dl.plan.profile_begin(K)
    uniq = [0] * len(dls)
    near = [0]

    def rec(li, dl, k):
        idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        nt = torch.empty(T, dtype=torch.int32, device=dev)
        dl.plan.debug_routing(dl.ws, T, idx, None, nt, stream=stream)
        uniq[li] += int(torch.unique(idx).numel())
        near[0] += int(nt.sum().item())

    for i in range(K):
        step(xs[W + i], routing=rec)
    torch.cuda.synchronize(dev)
    kt_all = {}
    for dl, _, _ in dls:
        for kname, (tms, n_l) in dl.plan.profile_end().items():
            a = kt_all.setdefault(kname, [0.0, 0])
            a[0] += tms
            a[1] += n_l
    alg_bytes = sum(uniq[li] * expert_bytes[li] for li in range(len(dls))) / K   # per step
    gu_ms, gu_n = kt_all.get("tc_gate_up", (0.0, 0))
    gu_bytes = sum(uniq[li] * expert_bytes[li] * 2 // 3 for li in range(len(dls))) / K
    pk = peaks()
    ach = (gu_bytes * K / gu_n) / (gu_ms / gu_n * 1e-3) / 1e9 if gu_n else None
    step_gbs = alg_bytes / (ms / K * 1e-3) / 1e9
    e2e_s, h2d, d2h = _e2e_steps(step, xs, K, W, (T, w.d), dev)
    e2e_s = max_over_ranks(e2e_s, dev)
    cpu = None
    if want_cpu and len(cpu_rates) == 2:
        per_tok_s = sum(3.0 / r for r in cpu_rates.values())
        cpu = {"value": 1.0 / per_tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": "oracle rate of one int4 and one int8 layer, combined as 3 + 3 layers per token "
                         "(RMSNorm is negligible); " + "; ".join(cpu_samples)}
    line = {
        "value": replica_tokens_per_s(world, K, T, ms), "unit": "tokens/s",
        "ms_per_step": ms / K, "hbm_gbs_layer": step_gbs, "hbm_frac_layer": step_gbs / pk["hbm_gbs"],
        "roofline": {"bound": "hbm", "kernel": "tc_gate_up", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": (ach / pk["hbm_gbs"]) if ach else None, "traffic": None, "peak_source": pk["source"],
                     "algorithmic_bytes_per_launch": gu_bytes / len(dls)},
        "kernel_ms_per_step": {k2: v[0] / K for k2, v in kt_all.items()},
        "e2e": {"value": world * K * T / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": K * sum(dl.plan.last_launch_count() + 1 for dl, _, _ in dls),
        "clocks": clocks,
        "routing": {"tokens": K * T * len(dls), "near_tie_tokens": near[0],
                    "unique_experts_per_step_per_layer": [u / K for u in uniq]},
        "config": workload_config(w, T, world),
        "cpu_baseline": cpu,
    }
    for dl, _, _ in dls:
        dl.close()
    del dls, xs
    torch.cuda.empty_cache()
    return line, gen_s


def bench_indexer(args, dev, world: int, want_cpu: bool, cpu_budget_s: float):
    """Sparse-attention key selection (lightning indexer scores + top-2048) for T query tokens at the end of
    a context of 65,536 cached keys.  Each step uses the key cache of the next of 16 layers (16 x 16.8 MB,
    larger than L2), as a decode step visits every layer's cache once."""
    import torch
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import to_dev

    w = H.INDEXER
    Ts = (args.tokens,) if args.tokens else w.T
    L = w.L
    n_sets = 16
    t0 = time.time()
    keys = [to_dev(w.keys(L, 100 + i), dev) for i in range(n_sets)]
    gen_s = time.time() - t0
    stream = torch.cuda.current_stream(dev)
    K, W = args.steps, args.warmup
    pk = peaks()
    frags = {}
    for T in Ts:
        qs = [to_dev(w.q(T, 1000 + i), dev) for i in range(K + W)]
        ws_ = [to_dev(w.w(T, 1000 + i), dev) for i in range(K + W)]
        nbytes = coli.colibri_indexer_workspace_size(T, L)
        wsp = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        out = torch.empty((T, w.topk), dtype=torch.int32, device=dev)
        state = {"i": 0}

        def step(i):
            coli.colibri_indexer_topk(T, L, L - T, w.H, w.d, w.topk, qs[i], ws_[i], keys[i % n_sets], out, wsp,
                                      nbytes, stream)
            return out

        def timed(fn):
            for i in range(W):
                fn(i)
            torch.cuda.synchronize(dev)
            if world > 1:
                torch.distributed.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(K):
                fn(W + i)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if world > 1:
                torch.distributed.barrier()
            return e0.elapsed_time(e1)

        with ClockSampler(dev.index) as clk:
            ms = timed(step)
        ms_sc = timed(lambda i: coli.colibri_indexer_scores(T, L, L - T, w.H, w.d, qs[i], ws_[i], keys[i % n_sets],
                                                            wsp, nbytes, stream))
        ms_sel = timed(lambda i: coli.colibri_indexer_select(T, L, L - T, w.topk, out, wsp, nbytes, stream))
        assert coli.colibri_indexer_check_status(wsp, stream) == 0
        # end to end: the query heads and weights from pinned host memory, the selection back
        qh = [qs[W + i].cpu().pin_memory() for i in range(K)]
        wh = [ws_[W + i].cpu().pin_memory() for i in range(K)]
        oh = torch.empty((K, T, w.topk), dtype=torch.int32).pin_memory()
        qd, wd = torch.empty_like(qs[0]), torch.empty_like(ws_[0])
        torch.cuda.synchronize(dev)
        te = time.perf_counter()
        for i in range(K):
            qd.copy_(qh[i], non_blocking=True)
            wd.copy_(wh[i], non_blocking=True)
            coli.colibri_indexer_topk(T, L, L - T, w.H, w.d, w.topk, qd, wd, keys[(W + i) % n_sets], out, wsp,
                                      nbytes, stream)
            oh[i].copy_(out, non_blocking=True)
        torch.cuda.synchronize(dev)
        e2e_s = max_over_ranks(time.perf_counter() - te, dev)
        ms, ms_sc, ms_sel = max_over_ranks(ms, dev), max_over_ranks(ms_sc, dev), max_over_ranks(ms_sel, dev)
        n_groups = (T + 3) // 4
        # algorithmic bytes of the score kernel(s): the keys once per launch group, the query heads and
        # weights, the scores written
        alg = n_groups * L * w.d * 2 + T * (w.H * w.d * 2 + w.H * 4) + T * L * 4
        ach = alg / (ms_sc / K * 1e-3) / 1e9
        cpu = None
        if want_cpu and T == Ts[0]:
            import oracle as O
            cores = O.default_threads()
            qc, wc, kc = w.q(1, 77), w.w(1, 77), w.keys(L, 77)
            tc0 = time.perf_counter()
            n = 0
            while time.perf_counter() - tc0 < cpu_budget_s:
                O.indexer_topk(O.indexer_scores(qc, wc, kc, L - 1, nthreads=cores), w.topk)
                n += 1
            dt = time.perf_counter() - tc0
            cpu = {"value": n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                   "sample": f"{n} query tokens over {L} keys (64 heads of 128, top-{w.topk}), fp64 scores over "
                             f"{cores} threads, {dt:.1f} s"}
        frags[T] = {
            "value": replica_tokens_per_s(world, K, T, ms), "unit": "tokens/s", "ms_per_step": ms / K,
            "roofline": {"bound": "hbm", "kernel": "indexer_scores", "achieved": ach, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
                         "traffic": INDEXER_SCORES_T1_TRAFFIC if (T == 1 and L == 65536) else None,
                         "duration": "the scores call: the 64-byte status clear and the kernel",
                         "peak_source": pk["source"],
                         "algorithmic_bytes_per_launch": alg},
            "kernel_ms_per_step": {"indexer_scores": ms_sc / K, "indexer_select": ms_sel / K},
            "e2e": {"value": world * K * T / e2e_s, "unit": "tokens/s",
                    "h2d_bytes_per_step": qh[0].numel() * qh[0].element_size() + wh[0].numel() * 4,
                    "d2h_bytes_per_step": T * w.topk * 4},
            "gpu_launches": K * (n_groups + 2),     # score kernel per group of 4 queries, mark, finish
            "clocks": clk.summary(),
            "config": {"workload": f"indexer: sparse-attention key selection (scores + top-{w.topk}) for T={T} "
                                   f"query tokens over {L} cached keys", "heads": w.H, "head_dim": w.d,
                       "topk": w.topk, "keys": L, "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": f"inputs larger than L2: {n_sets} key caches of {L * w.d * 2 / 1e6:.1f} MB cycled"},
            "cpu_baseline": cpu,
        }
    del keys
    torch.cuda.empty_cache()
    return frags, gen_s


def cpu_baseline(w, layer, T: int, budget_s: float):
    """The oracle as it stands on this host's cores (OpenMP over tokens), on a bounded sample of the
    workload's tokens: calls of `cores` tokens each until `budget_s` seconds have passed."""
    os.environ.setdefault("OMP_WAIT_POLICY", "PASSIVE")   # idle oracle threads sleep instead of spinning
    import oracle as O
    orc = O.Oracle(layer)
    cores = O.default_threads()
    n_tok = max(1, cores)
    x = w.x(max(T, n_tok), 77)
    toks = np.arange(n_tok, dtype=np.int32) % x.shape[0]
    t0 = time.perf_counter()
    done = 0
    while True:
        orc.forward(x, tokens=toks, nthreads=cores)
        done += n_tok
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} tokens of the {w.name} workload (d={w.d}, d_ff={w.F}, E={w.E}, k={w.k}"
                      f"{', shared d_ff=%d' % w.F_shared if w.F_shared else ''}), {n_tok} tokens per call over "
                      f"{cores} threads, {dt:.1f} s"}


def reference_arm(args, world: int, rank: int):
    """The oracle as it stands, timed on the host cores on the headline workload (decode, T=1)."""
    if rank != 0:
        return
    name = "decode" if args.workload == "all" else args.workload
    w, T_main, _ = workload_setup(name, args.experts, args.tokens)
    import oracle as O
    layer = w.layer(0)
    orc = O.Oracle(layer)
    cores = O.default_threads()
    n_tok = max(1, min(cores, 16))
    x = w.x(max(n_tok, T_main), 77)
    toks = np.arange(n_tok, dtype=np.int32) % x.shape[0]
    for _ in range(args.warmup):
        orc.forward(x, tokens=toks[:1], nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.forward(x, tokens=toks, nthreads=cores)
    dt = time.perf_counter() - t0
    v = args.steps * n_tok / dt
    sample = f"{n_tok} tokens per step of the {w.name} workload, {cores} threads"
    # n_gpus: the launch's N (the oracle itself runs on the host cores, as cpu_baseline says)
    print(json.dumps({"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
                      "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                      "data": "synthetic",
                      "config": workload_config(w, T_main, world),
                      "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                       "sample": sample},
                      "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


VARIANT_KEYS = ("value", "unit", "ms_per_step", "hbm_gbs_layer", "hbm_frac_layer", "roofline", "kernel_ms_per_step",
                "e2e", "gpu_launches", "clocks", "routing", "config", "cpu_baseline", "cache")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="all",
                    choices=["all", "decode", "mtp_verify", "prefill", "stacked", "indexer"],
                    help="all (default): decode T=1 as the headline with decode T=4, MTP verify, prefill and the "
                         "stacked layers as variants; otherwise that workload alone")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cache", action="store_true", help="skip the expert-cache variant of the decode workload")
    ap.add_argument("--no-idot", action="store_true", help="skip the integer-dot variants of decode and prefill")
    ap.add_argument("--experts", type=int, default=0, help="override E (reduced case for profiler captures)")
    ap.add_argument("--tokens", type=int, default=0, help="override T (reduced case for profiler captures)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, world, rank)
        return

    import torch
    import quantized_expert_ffn_bias_gb300 as coli
    coli.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    names = ["decode", "mtp_verify", "prefill", "stacked", "indexer"] if args.workload == "all" else [args.workload]
    results, gen_total = [], 0.0
    for name in names:
        budget = 10.0 if name == names[0] else 6.0
        if name == "indexer":
            frags, gen_s = bench_indexer(args, dev, world, want_cpu, budget)
            for T, fr in frags.items():
                results.append((f"indexer T={T}", "indexer", T, fr))
        elif name == "stacked":
            line, gen_s = bench_stacked(args, dev, world, want_cpu, budget)
            ws, T_s, _ = workload_setup("stacked", args.experts, args.tokens)
            results.append((f"stacked {ws.n_layers} layers T={T_s}", "stacked", None, line))
        else:
            frags, cpu, gen_s = bench_layer(name, args, dev, world, want_cpu, budget)
            for i, (T, fr) in enumerate(frags.items()):
                if T == "cache":
                    results.append(("decode T=1 with expert cache", name, 1, fr))
                    continue
                if T == "pilot":
                    results.append(("decode T=1, 2 layers, expert caches + next-layer prediction", name, 1, fr))
                    continue
                if isinstance(T, tuple):
                    results.append((f"{name} T={T[0]} integer-dot (IDOT)", name, T[0], fr))
                    continue
                fr["cpu_baseline"] = cpu if i == 0 else None
                results.append((f"{name} T={T}", name, T, fr))
        gen_total += gen_s
    if rank != 0:
        return
    head_label, head_name, head_T, head = results[0]
    line = {"metric": METRIC}
    line.update({k: head[k] for k in VARIANT_KEYS if k in head})
    if head_name == "indexer":
        dtype = "bf16 tensor-core operands, f32 accumulate"
    elif head_name == "stacked":
        dtype = "int4/int8-weights, fp16 tensor-core operands, f32 accumulate"
    elif head_T is not None and head_T > 8:
        dtype = "int4-weights, fp16 tensor-core operands, f32 accumulate"
    else:
        dtype = "int4-weights, int32 dot products, f32 accumulate"
    line.update({
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic (seeded; GLM-5.2-class shapes, random-init quantised experts)",
        "host_generation_s": round(gen_total, 1),
    })
    line["variants"] = {}
    for label, name, T, fr in results[1:]:
        line["variants"][label] = {k: fr[k] for k in VARIANT_KEYS if k in fr}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
