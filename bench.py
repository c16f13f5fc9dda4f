"""Benchmark of the verification step (verify attention over every layer + acceptance).

Default workload: Llama-3.1-8B-shaped, 32 layers of 32 query / 8 KV heads,
head_dim 128, bf16 KV cache of 122880 history tokens per layer (16.1 GB, read
once per step: larger than L2, so no flush is needed), gamma = 10 chain
(11 query tokens), acceptance over vocab 128256 with T = 1, eta = 1.

One JSON line on stdout (rank 0).  `value` = verify steps/s with all inputs
resident in HBM; `e2e` = the same through the public API with the per-step
inputs copied from pinned host memory and the results copied back inside the
timed region.  `--impl reference` times the double-precision CPU oracle on a
bounded sample of the same workload instead (it is the reference arm here).
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify-step KV-cache HBM GB/s vs GB300 peak; verify steps/s at 120K context"
UNIT = "verify_steps/s"
WORKLOAD = "llama3.1-8b_32layers_120k"
WORKLOAD_DEFAULT = WORKLOAD
# The traffic record is one 120K Llama-3.1-8B-shaped layer: the per-launch shape
# of these workloads.
TRAFFIC_WORKLOADS = ("llama3.1-8b_32layers_120k", "llama3.1-8b_1layer_120k")
L2_BYTES = 126 * 1024 * 1024   # the GB300 L2 (126 MiB)
SRC_FILES_TRAFFIC = ["long_context_speculative_gb300/csrc/attn_tc.cu",
                     "long_context_speculative_gb300/csrc/attn_simt.cu",
                     "long_context_speculative_gb300/csrc/attn.cuh",
                     "long_context_speculative_gb300/csrc/tcgen05.cuh",
                     "long_context_speculative_gb300/csrc/common.cuh"]


def max_over_ranks(dist, ms, device):
    """The slowest replica's time: the largest of every rank's `ms` (all ranks
    get it).  With no process group, `ms` itself."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world_size, steps, ms):
    """Steps of all replicas per second when each ran `steps` in at most `ms`."""
    return world_size * steps / (ms / 1e3)


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal (about 8 TB/s)

# NVML clock-event reason bits (nvml.h: nvmlClocksEventReason*)
_NVML_REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
                 0x4: "sw_power_cap"}


class NvmlClocks:
    """SM clock and clock-event reasons read through NVML (libnvidia-ml, the
    driver's own library, through ctypes) every `period_s` in a thread: fine
    enough to sample a timed region of a few tens of milliseconds."""

    def __init__(self, dev_index: int, period_s: float = 0.005):
        import ctypes
        self.ok = False
        self.samples = []
        self.period = period_s
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            found = False
            try:
                import torch
                uuid = str(torch.cuda.get_device_properties(dev_index).uuid)
                if not uuid.startswith("GPU-"):
                    uuid = "GPU-" + uuid
                found = nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
            except Exception:
                found = False
            if not found and nv.nvmlDeviceGetHandleByIndex_v2(dev_index, ctypes.byref(h)) != 0:
                return
            self.nv, self.h, self.ct = nv, h, ctypes
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None
            self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except Exception:
            self.ok = False

    def _run(self):
        ct = self.ct
        mhz = ct.c_uint()
        reasons = ct.c_ulonglong()
        while not self.stop:
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) == 0 and \
                    self.reasons_fn(self.h, ct.byref(reasons)) == 0:
                self.samples.append((float(mhz.value), int(reasons.value)))
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self.stop = False
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self.stop = True
            self.t.join(timeout=2)

    def summary(self):
        if not self.ok or not self.samples:
            return None
        sm = sorted(x for x, _ in self.samples)
        reasons = set()
        for _, bits in self.samples:
            for bit, name in _NVML_REASONS.items():
                if bits & bit:
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(sm), "source": f"NVML every {self.period * 1e3:.0f} ms"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region,
    with NVML sampled every 5 ms beside it (a timed region of a few tens of
    milliseconds gets only one or two nvidia-smi samples)."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.nvml = NvmlClocks(gpu_index)

    def __enter__(self):
        self.nvml.__enter__()
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.nvml.__exit__()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        nv = self.nvml.summary()
        smi = self.smi_summary()
        if nv is None:
            return smi
        # NVML's many samples decide the median; reasons seen by either count
        nv["reasons"] = sorted(set(nv["reasons"]) | set(r for r in smi["reasons"]
                                                       if r != "unavailable"))
        nv["nvidia_smi_samples"] = smi["samples"]
        return nv

    def smi_summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _traffic_for(kernel_key: str):
    """ncu DRAM bytes per launch from profiles/traffic.txt, if the kernel
    sources are unchanged since the capture (sha256 of its sources), else None."""
    try:
        rec = {}
        with open(os.path.join(ROOT, "profiles", "traffic.txt")) as f:
            for line in f:
                if line.startswith("#") or not line.strip():
                    continue
                k, v = line.split(None, 1)
                rec[k] = v.strip()
        if rec.get("key") != kernel_key or rec.get("src_sha256") != src_hash():
            return None
        return int(rec["dram_bytes_per_launch"])
    except Exception:
        return None


def src_hash():
    h = hashlib.sha256()
    for p in SRC_FILES_TRAFFIC:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline of our arm, and the whole reference arm)
# ---------------------------------------------------------------------------

def oracle_sample_time(w, layers_sample=1, groups_sample=1, seed=0):
    """Seconds per verify step of the oracle, from a bounded sample: the
    attention of `groups_sample` KV-head groups of `layers_sample` layers plus
    the full acceptance, scaled to all groups and layers."""
    import numpy as np
    import torch

    import oracle
    from long_context_speculative_gb300 import workloads as wl

    cores = oracle.default_threads()
    t_attn = 0.0
    rows_done = 0
    for layer in range(layers_sample):
        g = torch.Generator().manual_seed(seed + layer)
        G = w.G
        cap = w.capacity
        K = torch.randn((1, 1, cap, w.d), generator=g).to(torch.bfloat16)
        V = torch.randn((1, 1, cap, w.d), generator=g).to(torch.bfloat16)
        Q = torch.randn((1, G, w.n_q, w.d), generator=g).to(torch.bfloat16)
        pl = np.array([w.prefix], np.int32)
        for _ in range(groups_sample):
            t0 = time.perf_counter()
            oracle.verify_attn(wl.bf16_bits(Q), wl.bf16_bits(K), wl.bf16_bits(V), pl,
                               dtype=oracle.DTYPE_BF16, nthreads=cores)
            t_attn += time.perf_counter() - t0
            rows_done += G * w.n_q
    per_row = t_attn / rows_done
    attn_step = per_row * w.B * w.Hq * w.n_q * w.layers
    inp = wl.accept_inputs(w, B=1)
    t0 = time.perf_counter()
    oracle.accept(inp.z.numpy(), inp.q.numpy(), inp.tokens.numpy(), None, T=w.T, eta=w.eta,
                  seed=1, nthreads=cores)
    t_acc = time.perf_counter() - t0
    sample = (f"{layers_sample} layer x {groups_sample} of {w.Hkv} KV-head groups "
              f"({rows_done} query rows x {w.prefix} history rows, bf16 KV) + full acceptance "
              f"(11 x {w.V}); scaled to {w.layers} layers x {w.Hkv} groups")
    return attn_step + t_acc, cores, sample, t_attn + t_acc


def run_reference(args, w):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state; warm-up steps are free
    times = []
    sample = ""
    cores = 0
    work = 0.0
    for _ in range(args.steps):
        t, cores, sample, wall = oracle_sample_time(w)
        times.append(t)
        work += wall
    step_s = sum(times) / len(times)
    value = 1.0 / step_s
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers": w.layers, "context": w.prefix,
                       "n_q": w.n_q, "vocab": w.V, "l2": "inputs larger than L2"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, w):
    import torch

    from long_context_speculative_gb300 import rapid
    from long_context_speculative_gb300 import workloads as wl

    ws, rank, local = _dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    # ---- resident inputs: one KV cache and one Q per layer ------------------
    cap = w.capacity
    Ks, Vs, Qs = [], [], []
    mask = None
    prefix_len = None
    parents = None
    for layer in range(w.layers):
        a = wl.attn_inputs(w, layer=layer, device=dev)
        Ks.append(a.K); Vs.append(a.V); Qs.append(a.Q)
        if layer == 0:
            mask, prefix_len, parents = a.mask, a.prefix_len, a.parents
        del a
    acc_in = wl.accept_inputs(w, parents=parents if w.tree else None)
    z = acc_in.z.to(dev); q = acc_in.q.to(dev); tok = acc_in.tokens.to(dev)
    par = None if acc_in.parent is None else acc_in.parent.to(dev)
    # every layer's O and LSE in one tensor each, so that the end-to-end leg
    # reads them back with one copy apiece
    O_all = torch.empty((w.layers,) + tuple(Qs[0].shape), dtype=Qs[0].dtype, device=dev)
    L_all = torch.empty((w.layers, w.B, w.Hq, w.n_q), dtype=torch.float32, device=dev)
    Os = list(O_all.unbind(0))
    Ls = list(L_all.unbind(0))
    ws_attn = torch.empty(rapid.rapid_verify_attn_workspace_size(
        w.B, w.Hq, w.Hkv, w.d, w.n_q, cap, rapid.RAPID_DTYPE_BF16), dtype=torch.uint8, device=dev)
    ws_acc = torch.empty(rapid.rapid_accept_workspace_size(w.B, w.n_q, w.V), dtype=torch.uint8,
                         device=dev)
    n_acc = torch.empty(w.B, dtype=torch.int32, device=dev)
    nxt = torch.empty(w.B, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(seed, ev=None):
        for layer in range(w.layers):
            if ev is not None:
                ev[layer].record(stream)
            rapid.rapid_verify_attn(Qs[layer], Ks[layer], Vs[layer], prefix_len, mask, 0.0,
                                    Os[layer], Ls[layer], ws_attn)
        if ev is not None:
            ev[w.layers].record(stream)
        rapid.rapid_accept(z, q, tok, par, w.T, w.eta, seed, rapid.RAPID_ACCEPT_TAIL_CLAMP,
                           n_acc, nxt, None, None, ws_acc)

    for i in range(args.warmup):
        step(0x5EED0000 + i)
    torch.cuda.synchronize()
    assert rapid.rapid_device_error(True) == 0

    # ---- timed region (device-resident inputs): steps back to back, events
    # only around them (an event between two launches costs their overlap) ---
    start_ev = torch.cuda.Event(enable_timing=True)
    end_ev = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        start_ev.record(stream)
        for s in range(args.steps):
            step(0x5EED0000 + s)
        end_ev.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    total_ms = max_over_ranks(dist, start_ev.elapsed_time(end_ev), dev)
    assert rapid.rapid_device_error(True) == 0

    # ---- the same steps with an event around every rapid_verify_attn call:
    # the per-call time of the roofline (slightly pessimistic: the events keep
    # consecutive calls from overlapping) --------------------------------------
    roof_steps = min(args.steps, 20)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(w.layers + 1)]
           for _ in range(roof_steps)]
    for s in range(roof_steps):
        step(0x5EED1000 + s, evs[s])
    torch.cuda.synchronize()
    attn_ms = []
    for s in range(roof_steps):
        for layer in range(w.layers):
            attn_ms.append(evs[s][layer].elapsed_time(evs[s][layer + 1]))
    assert rapid.rapid_device_error(True) == 0

    # ---- e2e through the public API with host buffers -------------------------
    hQ = torch.empty((w.layers,) + tuple(Qs[0].shape), dtype=Qs[0].dtype).pin_memory()
    for layer in range(w.layers):
        hQ[layer].copy_(Qs[layer].cpu())
    hz = acc_in.z.clone().pin_memory(); hq = acc_in.q.clone().pin_memory()
    htok = acc_in.tokens.clone().pin_memory()
    hO = torch.empty((w.layers,) + tuple(Os[0].shape), dtype=Os[0].dtype).pin_memory()
    hL = torch.empty((w.layers,) + tuple(Ls[0].shape), dtype=torch.float32).pin_memory()
    hres = torch.empty(2 * w.B, dtype=torch.int32).pin_memory()
    dQ = torch.empty((w.layers,) + tuple(Qs[0].shape), dtype=Qs[0].dtype, device=dev)
    h2d = hQ.numel() * hQ.element_size() + hz.numel() * 4 + hq.numel() * 4 + htok.numel() * 4
    d2h = hO.numel() * hO.element_size() + hL.numel() * 4 + hres.numel() * 4
    res_dev = torch.empty(2 * w.B, dtype=torch.int32, device=dev)

    # The copies run on two copy streams beside the compute stream, within each
    # step: the step's inputs go up once the previous step's kernels are done
    # with the buffers (Q first, which the first layer waits for; z, q and the
    # tokens meanwhile, which only the acceptance waits for), and O and LSE of
    # every layer come back while the acceptance runs.  Nothing is enqueued
    # on the compute stream between two layers, so consecutive launches keep
    # their programmatic overlap.
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    ev_q = torch.cuda.Event()
    ev_zq = torch.cuda.Event()
    ev_attn = torch.cuda.Event()
    ev_res = torch.cuda.Event()
    ev_back = torch.cuda.Event()

    def e2e_step(seed, first):
        up.wait_stream(stream)   # the previous step's kernels are done with dQ, z, q, tok
        with torch.cuda.stream(up):
            dQ.copy_(hQ, non_blocking=True)
            ev_q.record(up)
            z.copy_(hz, non_blocking=True); q.copy_(hq, non_blocking=True)
            tok.copy_(htok, non_blocking=True)
            ev_zq.record(up)
        stream.wait_event(ev_q)
        if not first:
            stream.wait_event(ev_back)   # the previous step's results are out
        for layer in range(w.layers):
            rapid.rapid_verify_attn(dQ[layer], Ks[layer], Vs[layer], prefix_len, mask, 0.0,
                                    Os[layer], Ls[layer], ws_attn)
        ev_attn.record(stream)
        stream.wait_event(ev_zq)
        rapid.rapid_accept(z, q, tok, par, w.T, w.eta, seed, rapid.RAPID_ACCEPT_TAIL_CLAMP,
                           res_dev[:w.B], res_dev[w.B:], None, None, ws_acc)
        ev_res.record(stream)
        down.wait_event(ev_attn)
        with torch.cuda.stream(down):
            hO.copy_(O_all, non_blocking=True)
            hL.copy_(L_all, non_blocking=True)
        down.wait_event(ev_res)
        with torch.cuda.stream(down):
            hres.copy_(res_dev, non_blocking=True)
            ev_back.record(down)   # every result of this step is on the host

    for i in range(args.warmup):
        e2e_step(i, i == 0)
    torch.cuda.synchronize()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    up.wait_event(e_start)
    down.wait_event(e_start)
    for s in range(args.steps):
        e2e_step(0x5EED0000 + s, False)
    stream.wait_event(ev_back)   # the last step's results are on the host
    e_end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, e_start.elapsed_time(e_end), dev)

    # ---- rapid_accept alone on this step's own inputs (its share of a step) --
    acc_step_ms = accept_alone_ms(z, q, tok, par, w, ws_acc, n_acc, nxt, stream)

    # ---- acceptance bandwidth on batches larger than L2 ----------------------
    acc_roof = accept_batch_roofline(w, dev, stream)
    # and on the tree configuration's own step (4 x 32 rows of 152064 entries)
    acc_tree = None
    if not w.tree:
        acc_tree = accept_batch_roofline(wl.QWEN7B_TREE, dev, stream, B=wl.QWEN7B_TREE.B)
    # and on the same batch with drafts of different lengths (padding rows skipped)
    acc_ragged = accept_batch_roofline(w, dev, stream, ragged=True)
    # and on a batch large enough to amortise the per-call latency (128 sequences)
    acc_large = accept_batch_roofline(w, dev, stream, B=128)

    # ---- KV commit of an accepted path, all layers (moves the cache rows last) -
    kv_commit = kv_commit_timing(w, Ks, Vs, prefix_len, dev, stream)

    # ---- retrieval for the draft's context (once per request, not per step) -
    retrieval = retrieval_timing(w, dev, stream)

    # ---- target logits from the LM head, alone and followed by acceptance ---
    lm_head = lm_head_timing(w, dev, stream)

    # ---- numbers -----------------------------------------------------------
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(ws, args.steps, total_ms)
    e2e_value = whole_job_rate(ws, args.steps, e2e_ms)
    per_call = attn_call_bytes(w, prefix_len)
    attn_ms.sort()
    avg_call_ms = sum(attn_ms) / len(attn_ms)
    # The calls of the timed region run back to back, so the average call is
    # the step time less the acceptance's own share, over the layers.  The
    # event-bracketed pass after it keeps calls from overlapping and reads a
    # little slower; both are reported.
    step_call_ms = (ms_per_step - acc_step_ms) / w.layers
    achieved = per_call / (step_call_ms * 1e-3) / 1e9
    achieved_ev = per_call / (avg_call_ms * 1e-3) / 1e9
    peak, peak_src = _peaks()
    step_gbs = (per_call * w.layers + 2 * w.B * w.n_q * w.V * 4) / (ms_per_step * 1e-3) / 1e9
    launches_per_step = 2 * w.layers + 2
    step_kv = per_call * w.layers
    if step_kv > L2_BYTES:
        l2_note = f"inputs larger than L2 ({step_kv / 1e9:.2f} GB KV per step), no flush"
    else:
        l2_note = f"KV per step ({step_kv / 1e6:.1f} MB) fits in L2: not a bandwidth figure"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers": w.layers, "context": w.prefix,
                       "n_q": w.n_q, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "vocab": w.V,
                       "T": w.T, "eta": w.eta, "parallelism": f"replicas x{ws}",
                       "l2": l2_note},
            "kv_hbm_gbs_step": step_gbs,
            "roofline": {"bound": "hbm", "kernel": "rapid_verify_attn (history + merge kernels)",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                         "peak_source": peak_src + " (hbm_gbs, copy)",
                         "nominal_peak": NOMINAL_HBM_GBS,
                         "traffic": (_traffic_for("verify_attn_llama8b_120k")
                                     if w.name in TRAFFIC_WORKLOADS else None),
                         "algorithmic_bytes_per_launch": per_call,
                         "avg_launch_ms": step_call_ms,
                         "timing": (f"timed region: (ms_per_step {ms_per_step:.4f} - rapid_accept "
                                    f"alone on the step's inputs {acc_step_ms:.4f}) / "
                                    f"{w.layers} layers"),
                         "per_call_events": {
                             "avg_launch_ms": avg_call_ms, "achieved": achieved_ev,
                             "frac": achieved_ev / peak,
                             "frac_nominal": achieved_ev / NOMINAL_HBM_GBS,
                             "timing": f"CUDA events around every call, {roof_steps} steps "
                                       "after the timed region (calls cannot overlap)"}},
            "accept_step_ms": acc_step_ms,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "accept_roofline": acc_roof,
            "accept_roofline_tree": acc_tree,
            "accept_ragged": acc_ragged,
            "accept_roofline_large": acc_large,
            "kv_commit": kv_commit,
            "retrieval": retrieval,
            "lm_head_accept": lm_head,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
            "wall_s_timed": wall}
    # ---- the other workloads of the step, each timed the same way ----------
    del Ks, Vs, Qs, O_all, L_all, Os, Ls, dQ, hQ, hO, hL
    torch.cuda.empty_cache()
    if not args.no_extras and w.name == WORKLOAD_DEFAULT:
        line["extras"] = {x.name: extra_workload(x, dev, stream)
                          for x in (wl.LLAMA70B_128K, wl.QWEN7B_TREE, wl.LLAMA8B_DECODE_120K,
                                    wl.LLAMA1B_D64_120K)}
    if rank == 0 and not args.no_cpu_baseline:
        t, cores, sample, _ = oracle_sample_time(w, layers_sample=3, groups_sample=w.Hkv)
        line["cpu_baseline"] = {"value": 1.0 / t, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": sample}
        # the same oracle run on the bench's acceptance inputs: decisions and
        # tokens of the CUDA path against it, near-boundary cases counted
        line["parity_exemptions"] = parity_exemptions(w, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def attn_call_bytes(w, prefix_len):
    """Algorithmic bytes of one rapid_verify_attn call: K and V of the history
    and speculative rows read once per KV head, Q read, O and LSE written."""
    kv_rows = int(prefix_len.sum().item()) + w.B * w.n_q
    kv_bytes = 2 * w.Hkv * kv_rows * w.d * 2
    qo_bytes = 2 * w.B * w.Hq * w.n_q * w.d * 2 + w.B * w.Hq * w.n_q * 4
    return kv_bytes + qo_bytes


def accept_alone_ms(z, q, tok, par, w, ws_acc, n_acc, nxt, stream, reps=50):
    """Device time of one rapid_accept on a step's own inputs, back to back."""
    import torch

    from long_context_speculative_gb300 import rapid

    def call(seed):
        rapid.rapid_accept(z, q, tok, par, w.T, w.eta, seed, rapid.RAPID_ACCEPT_TAIL_CLAMP,
                           n_acc, nxt, None, None, ws_acc)

    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(reps):
        call(0x5EED2000 + i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def extra_workload(w, dev, stream, steps=10, warmup=3, roof_steps=5):
    """One more workload of the verify step, timed as the headline one: `steps`
    steps back to back (all layers of rapid_verify_attn, then rapid_accept),
    every call's share from the step time less the acceptance alone, and a
    pass with events around every call.  The caches exceed L2."""
    import torch

    from long_context_speculative_gb300 import rapid
    from long_context_speculative_gb300 import workloads as wl

    Ks, Vs, Qs = [], [], []
    for layer in range(w.layers):
        a = wl.attn_inputs(w, layer=layer, device=dev)
        Ks.append(a.K); Vs.append(a.V); Qs.append(a.Q)
        if layer == 0:
            mask, prefix_len, parents = a.mask, a.prefix_len, a.parents
        del a
    acc_in = wl.accept_inputs(w, parents=parents if w.tree else None)
    z, q, tok = acc_in.z.to(dev), acc_in.q.to(dev), acc_in.tokens.to(dev)
    par = None if acc_in.parent is None else acc_in.parent.to(dev)
    O = torch.empty_like(Qs[0])
    L = torch.empty((w.B, w.Hq, w.n_q), dtype=torch.float32, device=dev)
    ws_attn = torch.empty(rapid.rapid_verify_attn_workspace_size(
        w.B, w.Hq, w.Hkv, w.d, w.n_q, w.capacity, rapid.RAPID_DTYPE_BF16), dtype=torch.uint8,
        device=dev)
    ws_acc = torch.empty(rapid.rapid_accept_workspace_size(w.B, w.n_q, w.V), dtype=torch.uint8,
                         device=dev)
    n_acc = torch.empty(w.B, dtype=torch.int32, device=dev)
    nxt = torch.empty(w.B, dtype=torch.int32, device=dev)

    def step(seed, ev=None):
        for layer in range(w.layers):
            if ev is not None:
                ev[layer].record(stream)
            rapid.rapid_verify_attn(Qs[layer], Ks[layer], Vs[layer], prefix_len, mask, 0.0, O, L,
                                    ws_attn)
        if ev is not None:
            ev[w.layers].record(stream)
        rapid.rapid_accept(z, q, tok, par, w.T, w.eta, seed, rapid.RAPID_ACCEPT_TAIL_CLAMP,
                           n_acc, nxt, None, None, ws_acc)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(0x5EED0000 + i)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_step = e0.elapsed_time(e1) / steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(w.layers + 1)]
           for _ in range(roof_steps)]
    for i in range(roof_steps):
        step(0x5EED1000 + i, evs[i])
    torch.cuda.synchronize()
    per_ev = [evs[i][l].elapsed_time(evs[i][l + 1]) for i in range(roof_steps)
              for l in range(w.layers)]
    acc_ms = accept_alone_ms(z, q, tok, par, w, ws_acc, n_acc, nxt, stream)
    assert rapid.rapid_device_error(True) == 0
    per_call = attn_call_bytes(w, prefix_len)
    peak, _ = _peaks()
    call_ms = (ms_step - acc_ms) / w.layers
    ev_ms = sum(per_ev) / len(per_ev)
    gbs = per_call / (call_ms * 1e-3) / 1e9
    gbs_ev = per_call / (ev_ms * 1e-3) / 1e9
    out = {"verify_steps_per_s": 1e3 / ms_step, "ms_per_step": ms_step, "layers": w.layers,
           "B": w.B, "n_q": w.n_q, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
           "history": [int(x) for x in prefix_len.tolist()],
           "algorithmic_bytes_per_call": per_call, "accept_ms": acc_ms,
           "call_ms": call_ms, "achieved": gbs, "frac": gbs / peak,
           "frac_nominal": gbs / NOMINAL_HBM_GBS,
           "per_call_events": {"avg_launch_ms": ev_ms, "achieved": gbs_ev, "frac": gbs_ev / peak},
           "steps": steps, "unit": "GB/s"}
    del Ks, Vs, Qs
    torch.cuda.empty_cache()
    return out


def parity_exemptions(w, dev, B=16, seeds=4):
    """rapid_accept on B sequences of the bench's acceptance inputs against the
    oracle on the same inputs, for a few Philox keys: decisions and tokens must
    agree except in the stated near-boundary bands, whose cases are counted
    (oracle.parity.accept_exemptions)."""
    import torch

    import oracle
    from oracle.parity import accept_exemptions
    from long_context_speculative_gb300 import rapid
    from long_context_speculative_gb300 import workloads as wl

    inp = wl.accept_inputs(w, B=B)
    zn, qn, tn = inp.z.numpy(), inp.q.numpy(), inp.tokens.numpy()
    pn = None if inp.parent is None else inp.parent.numpy()
    z, q, tok = inp.z.to(dev), inp.q.to(dev), inp.tokens.to(dev)
    par = None if inp.parent is None else inp.parent.to(dev)
    tot = {}
    for k in range(seeds):
        seed = 0x5EED3000 + k
        res = rapid.accept(z, q, tok, par, T=w.T, eta=w.eta, seed=seed)
        torch.cuda.synchronize()
        g = {key: v.cpu().numpy() for key, v in res.items()}
        r = oracle.accept(zn, qn, tn, pn, T=w.T, eta=w.eta, seed=seed)
        for key, v in accept_exemptions(zn, qn, tn, pn, w.T, w.eta, True, g, r).items():
            tot[key] = tot.get(key, 0) + v
    tot["batch"] = f"{B} x {w.n_q} x {w.V}, {seeds} Philox keys, T = {w.T}, eta = {w.eta}"
    return tot


def kv_commit_timing(w, Ks, Vs, prefix_len, dev, stream, reps=20):
    """rapid_kv_commit over every layer for an accepted path that moves rows
    (nodes 2, 4, 6, ...: every destination differs from its source).  The
    moved bytes are tiny, so this is a latency figure, not a bandwidth one:
    through the Python binding call by call (a KVLayerTable packs the layer
    pointers once), and as device time from a CUDA graph of the same calls."""
    import torch

    from long_context_speculative_gb300 import rapid

    n = (w.n_q - 1) // 2
    path = torch.full((w.B, w.n_q), -1, dtype=torch.int32)
    if n > 0:
        path[:, :n] = torch.arange(2, 2 * n + 1, 2, dtype=torch.int32)
    path = path.to(dev)
    n_acc = torch.full((w.B,), n, dtype=torch.int32, device=dev)

    table = rapid.KVLayerTable(Ks, Vs)

    def call():
        table.commit(prefix_len, path, n_acc)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    eager_us = e0.elapsed_time(e1) / reps * 1e3
    if n == 0:   # a single-query step has no speculative rows: the call launches nothing
        return {"us_per_step": eager_us, "us_per_step_graph": None, "layers": w.layers,
                "rows_moved_per_layer": 0, "bytes_moved": 0, "launches_per_step": 0}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(reps):
            call()
    graph.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0.record(cur)
    graph.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    graph_us = e0.elapsed_time(e1) / reps * 1e3
    assert rapid.rapid_device_error(True) == 0
    moved = w.layers * w.B * w.Hkv * n * w.d * 2 * 2   # K and V rows, bf16
    return {"us_per_step": eager_us, "us_per_step_graph": graph_us, "layers": w.layers,
            "rows_moved_per_layer": w.B * w.Hkv * n, "bytes_moved": moved,
            "launches_per_step": 1}


def lm_head_timing(w, dev, stream, hidden=4096, reps=20):
    """rapid_lm_head and rapid_lm_head_accept for the workload's verify rows
    (B * n_q hidden states of width 4096, a V x 4096 bf16 head: 1.05 GB for
    the 128256-entry vocabulary, larger than L2, so every call streams it from
    HBM).  Algorithmic bytes = W + hidden states read once + z written."""
    import torch

    from long_context_speculative_gb300 import rapid
    from long_context_speculative_gb300 import workloads as wl

    rows = w.B * w.n_q
    if rows > rapid.RAPID_LM_HEAD_MAX_ROWS:
        return {"skipped": f"{rows} verify rows > {rapid.RAPID_LM_HEAD_MAX_ROWS}"}
    g = torch.Generator(device=dev).manual_seed(4096)
    H = torch.randn((rows, hidden), generator=g, device=dev).to(torch.bfloat16)
    W = torch.empty((w.V, hidden), dtype=torch.bfloat16, device=dev)
    for i in range(0, w.V, 16384):   # fill in slices to bound the fp32 temporary
        n = min(16384, w.V - i)
        W[i:i + n] = (torch.randn((n, hidden), generator=g, device=dev) * (3.0 / 64)).to(torch.bfloat16)
    z = torch.empty((rows, w.V), dtype=torch.float32, device=dev)
    inp = wl.accept_inputs(w)
    q, tok = inp.q.to(dev), inp.tokens.to(dev)
    par = None if inp.parent is None else inp.parent.to(dev)
    ws = torch.empty(rapid.rapid_lm_head_accept_workspace_size(w.B, w.n_q, w.V), dtype=torch.uint8,
                     device=dev)
    n_acc = torch.empty(w.B, dtype=torch.int32, device=dev)
    nxt = torch.empty(w.B, dtype=torch.int32, device=dev)

    def fused(i):
        rapid.rapid_lm_head_accept(H, W, q, tok, par, w.T, w.eta, i,
                                   rapid.RAPID_ACCEPT_TAIL_CLAMP, n_acc, nxt, None, None, ws)

    for i in range(3):
        rapid.rapid_lm_head(H, W, z)
        fused(i)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    ev[0].record(stream)
    for _ in range(reps):
        rapid.rapid_lm_head(H, W, z)
    ev[1].record(stream)
    for i in range(reps):
        fused(100 + i)
    ev[2].record(stream)
    torch.cuda.synchronize()
    assert rapid.rapid_device_error(True) == 0
    ms_head = ev[0].elapsed_time(ev[1]) / reps
    ms_fused = ev[1].elapsed_time(ev[2]) / reps
    nbytes = W.numel() * 2 + H.numel() * 2 + z.numel() * 4
    peak, _ = _peaks()
    gbs = nbytes / (ms_head * 1e-3) / 1e9
    out = {"rows": rows, "hidden": hidden, "vocab": w.V, "weight_bytes": W.numel() * 2,
           "lm_head_us": ms_head * 1e3, "lm_head_accept_us": ms_fused * 1e3,
           "roofline": {"bound": "hbm", "kernel": "lm_head_kernel", "achieved": gbs, "peak": peak,
                        "unit": "GB/s", "frac": gbs / peak, "algorithmic_bytes_per_launch": nbytes}}
    del W
    torch.cuda.empty_cache()
    return out


def retrieval_timing(w, dev, stream, D=1024, reps=20):
    """Chunk scoring and budgeted selection for the draft's retrieved context:
    chunks of 512 tokens of the workload's context, 1024-wide bf16 embeddings.
    One request (device time of both calls) and a batch of requests whose
    chunk embeddings exceed L2 (scores: algorithmic bytes = the embeddings read
    once + the scores written, / CUDA-event time per call).  Calls are replayed
    from a CUDA graph, so host launch cost is not in the figures."""
    import torch

    from long_context_speculative_gb300 import rapid

    N = -(-w.prefix // 512)
    out = {"chunks_per_request": N, "embed_dim": D, "dtype": "bf16"}
    g = torch.Generator().manual_seed(2024)

    def run(Bq):
        q = torch.randn((Bq, D), generator=g).to(torch.bfloat16).to(dev)
        c = torch.randn((Bq, N, D), generator=g).to(torch.bfloat16).to(dev)
        ctx = torch.full((Bq,), w.prefix, dtype=torch.int32, device=dev)
        s = torch.empty((Bq, N), dtype=torch.float32, device=dev)
        sel = torch.empty((Bq, N), dtype=torch.int32, device=dev)
        ns = torch.empty(Bq, dtype=torch.int32, device=dev)
        ts = torch.empty(Bq, dtype=torch.int32, device=dev)

        def scores_call():
            rapid.rapid_retrieval_scores(q, c, s)

        def select_call():
            rapid.rapid_retrieval_select(s, ctx, sel, ns, ts, threshold=-1.0)

        for _ in range(3):
            scores_call()
            select_call()
        torch.cuda.synchronize()
        # each call's kernels are tiny for one request: replay a CUDA graph of
        # `reps` calls so that the host's launch cost is not in the figure
        out_ms = []
        for fn in (scores_call, select_call):
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(reps):
                    fn()
            graph.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            cur = torch.cuda.current_stream()
            e0.record(cur)
            graph.replay()
            e1.record(cur)
            torch.cuda.synchronize()
            out_ms.append(e0.elapsed_time(e1) / reps)
        assert rapid.rapid_device_error(True) == 0
        return out_ms[0], out_ms[1], c.numel() * 2 + q.numel() * 2 + s.numel() * 4

    ms_s, ms_sel, _ = run(1)
    out["request_us"] = {"scores": ms_s * 1e3, "select": ms_sel * 1e3}
    Bq = max(1, -(-200_000_000 // (N * D * 2)))
    ms_s, ms_sel, nbytes = run(Bq)
    peak, peak_src = _peaks()
    gbs = nbytes / (ms_s * 1e-3) / 1e9
    out["batch"] = {"requests": Bq, "scores_ms": ms_s, "select_ms": ms_sel,
                    "scores_roofline": {"bound": "hbm", "achieved": gbs, "peak": peak,
                                        "unit": "GB/s", "frac": gbs / peak,
                                        "algorithmic_bytes_per_launch": nbytes}}
    return out


def _device_accept_inputs(w, B, dev):
    """The acceptance inputs of workloads.accept_inputs (z ~ N(0, z_std^2),
    q = softmax(z/T + noise), each draft token drawn from q of its parent's
    row), generated on the device for batches too large to build on the host."""
    import torch

    from long_context_speculative_gb300 import workloads as wl

    g = torch.Generator(device=dev).manual_seed(w.seed * 7919 + 77)
    z = torch.randn((B, w.n_q, w.V), generator=g, device=dev) * w.z_std
    base = z / w.T if w.q_noise_uses_T else z
    q = torch.softmax(base + torch.randn((B, w.n_q, w.V), generator=g, device=dev)
                      * w.q_noise_std, dim=-1)
    if w.tree:
        gt = wl.gen(w.seed * 7919 + 11)
        parents = torch.tensor([wl.random_tree(w.n_q, w.tree_nodes_max_depth, gt)
                                for _ in range(B)], dtype=torch.int64)
    else:
        parents = torch.tensor([wl.chain_parents(w.n_q)] * B, dtype=torch.int64)
    rows = parents[:, 1:].clamp(min=0).to(dev)                    # parent row of nodes 1..n_q-1
    src = torch.gather(q, 1, rows[:, :, None].expand(B, w.n_q - 1, w.V))
    tok = torch.zeros((B, w.n_q), dtype=torch.int32, device=dev)
    tok[:, 1:] = torch.multinomial(src.reshape(-1, w.V), 1, generator=g).view(B, w.n_q - 1).int()
    par = None
    if w.tree:
        par = parents.to(torch.int32)
        par[:, 0] = -1
        par = par.to(dev)
    return z.contiguous(), q.contiguous(), tok, par


def accept_batch_roofline(w, dev, stream, reps=20, B=None, ragged=False):
    """rapid_accept alone on a batch of at least 100 MB of z + q (larger than L2):
    the workload's own batch when that is large enough (the 4-sequence tree of
    the Qwen shape: 155.7 MB), else 16 sequences of its rows, more if that stays
    under 100 MB.  Algorithmic bytes = 8 B per vocabulary entry (z and q read
    once) / CUDA-event time per call.  ragged: the same batch with seeded draft
    lengths 1..n_q per sequence (rapid_accept_ex); only the real rows count."""
    import torch

    from long_context_speculative_gb300 import rapid
    from long_context_speculative_gb300 import workloads as wl

    if B is not None:
        Bb = B
    elif w.B * w.n_q * w.V * 8 >= 100_000_000:
        Bb = w.B
    else:
        Bb = max(16, -(-100_000_000 // (w.n_q * w.V * 8)))
    if Bb * w.n_q * w.V * 8 > 1_000_000_000:
        z, q, tok, par = _device_accept_inputs(w, Bb, dev)
    else:
        inp = wl.accept_inputs(w, B=Bb)
        z, q, tok = inp.z.to(dev), inp.q.to(dev), inp.tokens.to(dev)
        par = None if inp.parent is None else inp.parent.to(dev)
    nbytes = z.numel() * 4 + q.numel() * 4
    nn = None
    if ragged:
        g = torch.Generator().manual_seed(w.seed + 404)
        counts = torch.randint(1, w.n_q + 1, (Bb,), generator=g, dtype=torch.int32)
        nn = counts.to(dev)
        nbytes = int(counts.sum()) * w.V * 8
    ws = torch.empty(rapid.rapid_accept_workspace_size(Bb, w.n_q, w.V), dtype=torch.uint8,
                     device=dev)
    na = torch.empty(Bb, dtype=torch.int32, device=dev)
    nt = torch.empty(Bb, dtype=torch.int32, device=dev)

    def call(seed):
        if nn is None:
            rapid.rapid_accept(z, q, tok, par, w.T, w.eta, seed, rapid.RAPID_ACCEPT_TAIL_CLAMP,
                               na, nt, None, None, ws)
        else:
            rapid.rapid_accept_ex(z, q, tok, par, nn, w.T, w.eta, seed,
                                  rapid.RAPID_ACCEPT_TAIL_CLAMP, na, nt, None, None, ws)

    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(reps):
        call(100 + i)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    # the same calls replayed from a CUDA graph (no host launch cost between them)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(reps):
            call(200 + i)
    graph.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_graph = e0.elapsed_time(e1) / reps
    achieved = nbytes / (ms * 1e-3) / 1e9
    peak, src = _peaks()
    if nn is None:
        batch = f"{Bb} x {w.n_q} x {w.V} fp32 z and q ({nbytes / 1e6:.1f} MB, > L2)"
    else:
        batch = (f"{Bb} x {w.n_q} x {w.V} fp32 z and q, draft lengths 1..{w.n_q} "
                 f"({int(counts.sum())} real rows: {nbytes / 1e6:.1f} MB)")
    return {"bound": "hbm", "kernel": "rapid_accept (row + select kernels)",
            "batch": batch,
            "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "avg_launch_ms": ms, "avg_launch_ms_graph": ms_graph,
            "peak_source": src + " (hbm_gbs, copy)"}


def profile_accept(w, B):
    """Three rapid_accept calls on B sequences of w (chain or tree as w is), no timing."""
    import torch

    from long_context_speculative_gb300 import rapid
    from long_context_speculative_gb300 import workloads as wl

    inp = wl.accept_inputs(w, B=B)
    dev = torch.device("cuda:0")
    z, q, tok = inp.z.to(dev), inp.q.to(dev), inp.tokens.to(dev)
    par = None if inp.parent is None else inp.parent.to(dev)
    for i in range(3):
        rapid.accept(z, q, tok, par, T=w.T, eta=w.eta, seed=i)
    torch.cuda.synchronize()
    err = rapid.rapid_device_error()
    print(json.dumps({"profile_accept": B, "rows": B * w.n_q, "vocab": w.V, "device_error": err}))
    if err:
        sys.exit(1)


def profile_lm_head(rows=11, hidden=4096, V=128256):
    """Three rapid_lm_head calls (11 rows x 4096 against a 128256 x 4096 bf16 head), no timing."""
    import torch

    from long_context_speculative_gb300 import rapid

    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(4096)
    H = torch.randn((rows, hidden), generator=g, device=dev).to(torch.bfloat16)
    W = torch.empty((V, hidden), dtype=torch.bfloat16, device=dev)
    for i in range(0, V, 16384):
        n = min(16384, V - i)
        W[i:i + n] = (torch.randn((n, hidden), generator=g, device=dev) * (3.0 / 64)).to(torch.bfloat16)
    z = torch.empty((rows, V), dtype=torch.float32, device=dev)
    for _ in range(3):
        rapid.rapid_lm_head(H, W, z)
    torch.cuda.synchronize()
    err = rapid.rapid_device_error()
    print(json.dumps({"profile_lm_head": rows, "hidden": hidden, "vocab": V, "device_error": err}))
    if err:
        sys.exit(1)


def profile_lm_head_accept(rows=11, hidden=4096, V=128256):
    """Three rapid_lm_head_accept calls of one 11-row chain step (the single
    fused kernel) against a 128256 x 4096 bf16 head, no timing."""
    import torch

    from long_context_speculative_gb300 import rapid
    from long_context_speculative_gb300 import workloads as wl

    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(4096)
    H = torch.randn((rows, hidden), generator=g, device=dev).to(torch.bfloat16)
    W = torch.empty((V, hidden), dtype=torch.bfloat16, device=dev)
    for i in range(0, V, 16384):
        n = min(16384, V - i)
        W[i:i + n] = (torch.randn((n, hidden), generator=g, device=dev) * (3.0 / 64)).to(torch.bfloat16)
    inp = wl.accept_inputs(wl.LLAMA8B_120K)
    q, tok = inp.q.to(dev), inp.tokens.to(dev)
    for i in range(3):
        rapid.lm_head_accept(H, W, q, tok, None, T=1.0, eta=1.0, seed=i)
    torch.cuda.synchronize()
    err = rapid.rapid_device_error()
    print(json.dumps({"profile_lm_head_accept": rows, "hidden": hidden, "vocab": V,
                      "device_error": err}))
    if err:
        sys.exit(1)


def profile_retrieval(B, N=240, D=1024):
    """Three scores + select calls on B requests of N chunks x D bf16, no timing."""
    import torch

    from long_context_speculative_gb300 import rapid

    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(2024)
    q = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    c = torch.randn((B, N, D), generator=g).to(torch.bfloat16).to(dev)
    ctx = torch.full((B,), N * 512, dtype=torch.int32, device=dev)
    s = torch.empty((B, N), dtype=torch.float32, device=dev)
    sel = torch.empty((B, N), dtype=torch.int32, device=dev)
    ns = torch.empty(B, dtype=torch.int32, device=dev)
    ts = torch.empty(B, dtype=torch.int32, device=dev)
    for _ in range(3):
        rapid.rapid_retrieval_scores(q, c, s)
        rapid.rapid_retrieval_select(s, ctx, sel, ns, ts, threshold=-1.0)
    torch.cuda.synchronize()
    err = rapid.rapid_device_error()
    print(json.dumps({"profile_retrieval": B, "chunks": N, "dim": D, "device_error": err}))
    if err:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the 70B, tree, decode and d=64 workloads after the headline one")
    ap.add_argument("--workload", default=None,
                    help="named workload (default: the 32-layer 120K Llama-3.1-8B step)")
    ap.add_argument("--profile-lm-head", action="store_true",
                    help="run rapid_lm_head three times on 11 x 4096 rows against a "
                         "128256 x 4096 head (for ncu) and exit")
    ap.add_argument("--profile-lm-head-accept", action="store_true",
                    help="run rapid_lm_head_accept three times on one 11-row step against a "
                         "128256 x 4096 head (for ncu) and exit")
    ap.add_argument("--profile-retrieval", type=int, default=0, metavar="B",
                    help="run retrieval scores + select on B requests of 240 chunks x 1024 "
                         "(for ncu) and exit")
    ap.add_argument("--profile-accept", type=int, default=0, metavar="B",
                    help="only run rapid_accept three times on B sequences of the "
                         "workload's rows (a fixed launch sequence for ncu captures)")
    args = ap.parse_args()
    from long_context_speculative_gb300 import workloads as wl
    w = wl.LLAMA8B_120K
    if args.workload is not None:
        w = {x.name: x for x in wl.ALL}[args.workload]
    global WORKLOAD
    WORKLOAD = w.name
    if args.profile_lm_head:
        profile_lm_head()
        return
    if args.profile_lm_head_accept:
        profile_lm_head_accept()
        return
    if args.profile_retrieval > 0:
        profile_retrieval(args.profile_retrieval)
        return
    if args.profile_accept > 0:
        profile_accept(w, args.profile_accept)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
