"""Benchmark: routed-expert MoE decode on one GB300 (or N replicas under torchrun).

Default workload (the headline line): the Qwen3-30B-A3B-shaped NVFP4 decode
layer -- H=2048, I=768, E=128 experts, top-8, T=1 token -- as a stack of 48
distinct resident layer banks (48 x 340 MB, far beyond the 129 MB L2), each
with its own softmax top-8 routing of N(0,1) logits.  One step = one token
through all 48 layers (48 moe_decode calls, one fused kernel each at T=1),
replayed from one CUDA graph.  value = layer-tokens/s (tokens x layers / s).

Also reported in the same line: the 47-layer Laguna-shaped stack (39 Q4_K +
8 BF16 layers, H=4096, I=768, E=256, top-10, Zipf(1.1) routing, 85.4 GiB
resident) at T = 1, 4, 16, 64 as stack tokens/s, and the NVFP4 layer at T=8.

Also reported: the prompt path (moe_prefill_grouped) on a 4096-token chunk of
the same NVFP4 layer, W4A4 and W4A8, as tokens/s and tensor TFLOP/s.

Roofline: the timed unit is one moe_decode pass (at T=1 one k_layer_small
launch); achieved GB/s =
the algorithmic bytes of a pass (each routed expert's gate_up and down rows
once, plus x, ids, weights and out) / the pass's average duration from CUDA
events on the launching stream.  Peak = MEASURED_PEAKS.json hbm_gbs.

--impl reference times the CPU oracle (numpy, fp64) on a bounded sample of
the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

NVFP4, Q4_K, BF16, Q8_0, Q6_K, Q4_0 = 3, 2, 0, 1, 4, 5
TYPE_NAMES = {BF16: "bf16", Q8_0: "q8_0", Q4_K: "q4_k", NVFP4: "nvfp4", Q6_K: "q6_k", Q4_0: "q4_0"}
CFG1 = dict(H=2048, I=768, E=128, K=8, gu=NVFP4, dn=NVFP4)
LAGUNA = dict(H=4096, I=768, E=256, K=10)
# the other GGUF row types at the same layer shape as the headline (gate_up, down)
TYPE_PAIRS = ((Q4_K, Q6_K), (Q6_K, Q6_K), (Q4_0, Q4_0), (Q8_0, Q8_0), (Q4_K, Q4_K))


def row_bytes(t, k):
    return {0: 2 * k, 1: k // 32 * 34, 2: k // 256 * 144, 3: k // 2 + k // 16, 4: k // 256 * 210,
            5: k // 32 * 18}[t]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """SM clock and throttle reasons sampled during the timed region: NVML read
    through ctypes about every millisecond (the GPU found by its UUID, so the
    right one of a shared machine's GPUs), else nvidia-smi every 20 ms.  Read
    only; no setting is changed."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []          # (sm_mhz, max_mhz, reason names)
        self.proc = None
        self.stop = threading.Event()
        self.thread = None
        self.source = None

    def _nvml_handle(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return None, None
        h = ctypes.c_void_p()
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.gpu).uuid)
            key = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if nv.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(h)) == 0:
                return nv, h
        except Exception:
            pass
        return None, None

    def _nvml_loop(self, nv, h):
        import ctypes
        sm, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        try:
            get_reasons = nv.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            get_reasons = nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0:
                names = []
                if get_reasons(h, ctypes.byref(rs)) == 0:
                    names = [n for n, b in self.REASONS.items() if rs.value & b]
                self.rows.append((float(sm.value), float(mx.value), names))
            time.sleep(0.001)

    def __enter__(self):
        try:
            nv, h = self._nvml_handle()
        except OSError:
            nv, h = None, None
        if nv is not None:
            self.source = "nvml, ~1 ms"
            self.thread = threading.Thread(target=self._nvml_loop, args=(nv, h), daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, 20 ms"
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None
        return self

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            r = [c.strip() for c in line.split(",")]
            if len(r) > 8 and r[1].replace(".", "").isdigit() and r[2].replace(".", "").isdigit():
                self.rows.append((float(r[1]), float(r[2]),
                                  [n for n, v in zip(names, r[5:9]) if v.lower() == "active"]))

    def __exit__(self, *a):
        self.stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [r[0] for r in self.rows]
        reasons = sorted({n for r in self.rows for n in r[2]})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r[1] for r in self.rows),
                "reasons": reasons, "samples": len(self.rows), "source": self.source}


# ------------------------------------------------------------------ stacks of layers on the device

class Stack:
    """NL resident layers (banks on the device) plus, after ``prepare``, the
    inputs/outputs of one batch size and a captured CUDA graph of one step."""

    def __init__(self, layer_types, H, I, E, K, seed, dev):
        import torch

        from quantized_routed_expert_route_gb300 import capi
        from synth import banks as S
        from synth import counter as C
        self.torch, self.capi, self.S, self.dev = torch, capi, S, dev
        self.H, self.I, self.E, self.K = H, I, E, K
        self.NL = len(layer_types)
        self.layers = []
        stream = torch.cuda.current_stream().cuda_stream
        for l, (gu_t, dn_t) in enumerate(layer_types):
            rb_gu, rb_dn = row_bytes(gu_t, H), row_bytes(dn_t, I)
            gu = torch.empty(E * 2 * I * rb_gu + 16, dtype=torch.uint8, device=dev)
            dn = torch.empty(E * H * rb_dn + 16, dtype=torch.uint8, device=dev)
            C.fill_bank_torch(gu[: E * 2 * I * rb_gu], seed * 1000 + 2 * l, gu_t, H)
            C.fill_bank_torch(dn[: E * H * rb_dn], seed * 1000 + 2 * l + 1, dn_t, I)
            sb = torch.from_numpy(S.counter_scale_bank(seed * 1000 + l, E, gu_t, dn_t)).to(dev)
            geom = capi.moe_layer_geom(H, I, E, K, gu_t, dn_t)
            bank = capi.moe_bank_create(geom, gu.data_ptr(), E * 2 * I * rb_gu, dn.data_ptr(), E * H * rb_dn,
                                        sb.data_ptr(), capi.MOE_SRC_DEVICE_BORROW, stream)
            self.layers.append(dict(gu=gu, dn=dn, sb=sb, bank=bank, expert_bytes=2 * I * rb_gu + H * rb_dn))
        self.graph = None
        self.stream = torch.cuda.Stream(device=dev)

    def prepare(self, T, routing, seed):
        torch, capi, S = self.torch, self.capi, self.S
        self.T = T
        self.bytes_per_step = 0
        self.unique_per_layer = []
        for l, L in enumerate(self.layers):
            if routing == "zipf":
                ids, w = S.zipf_routing(seed * 7 + l, T, self.E, self.K)
            else:
                ids, w = S.softmax_topk_routing(seed * 7 + l, T, self.E, self.K)
            uniq = len(np.unique(ids))
            self.unique_per_layer.append(uniq)
            self.bytes_per_step += uniq * L["expert_bytes"] + T * self.H * 2 * 2 + T * self.K * 8
            L["ids"] = torch.from_numpy(ids).to(self.dev)
            L["w"] = torch.from_numpy(w).to(self.dev)
        self.ws_bytes = max(capi.moe_workspace_bytes(L["bank"], T) for L in self.layers)
        self.launches_per_step = sum(capi.moe_decode_kernel_count(L["bank"], T) for L in self.layers)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.dev)
        capi.moe_workspace_init(self.ws.data_ptr(), self.ws_bytes, torch.cuda.current_stream().cuda_stream)
        g = np.random.default_rng(seed)
        xs = torch.from_numpy(g.standard_normal((self.NL, T, self.H)).astype(np.float32))
        self.x = xs.to(torch.bfloat16).to(self.dev)
        self.out = torch.empty((self.NL, T, self.H), dtype=torch.bfloat16, device=self.dev)
        self.graph = None
        self.capture()

    def launch_all(self, stream_ptr):
        capi = self.capi
        for l, L in enumerate(self.layers):
            capi.moe_decode(L["bank"], self.x[l].data_ptr(), self.T, L["ids"].data_ptr(), L["w"].data_ptr(),
                            self.out[l].data_ptr(), self.ws.data_ptr(), self.ws_bytes, stream_ptr)

    def capture(self):
        torch = self.torch
        s = self.stream
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.launch_all(s.cuda_stream)
            s.synchronize()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=s):
                self.launch_all(s.cuda_stream)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()

    def time_replays(self, steps, warmup):
        torch = self.torch
        s = self.stream
        with torch.cuda.stream(s):
            for _ in range(warmup):
                self.graph.replay()
            s.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(steps):
                self.graph.replay()
            e1.record(s)
            e1.synchronize()
        return e0.elapsed_time(e1) / steps   # ms per step

    def time_e2e(self, steps, warmup):
        """End to end through the C ABI's host-buffer entry point: per step,
        every layer's moe_decode_host copies its x, ids and weights from
        pinned host memory (laid out as the library's staging layout, so one
        copy carries all three), decodes and copies its output back to pinned
        host memory (48 calls captured in one CUDA graph); the step ends when
        the host has the outputs."""
        torch, capi = self.torch, self.capi
        s = self.stream
        T, K, H = self.T, self.K, self.H
        iob = max(capi.moe_decode_io_bytes(L["bank"], T) for L in self.layers)
        o_ids, o_w, _ = capi.moe_decode_io_offsets(self.layers[0]["bank"], T)
        hin = torch.zeros((self.NL, iob), dtype=torch.uint8).pin_memory()
        for l, L in enumerate(self.layers):
            hin[l, : 2 * T * H] = self.x[l].cpu().view(torch.uint8).reshape(-1)
            hin[l, o_ids: o_ids + 4 * T * K] = L["ids"].cpu().view(torch.uint8).reshape(-1)
            hin[l, o_w: o_w + 4 * T * K] = L["w"].cpu().view(torch.uint8).reshape(-1)
        hout = [torch.empty((T, H), dtype=torch.int16).pin_memory() for _ in range(self.NL)]
        io = torch.empty((self.NL, iob), dtype=torch.uint8, device=self.dev)
        h2d = self.NL * (o_w + 4 * T * K)
        d2h = sum(t.numel() * 2 for t in hout)

        def launch(sp):
            for l, L in enumerate(self.layers):
                base = hin[l].data_ptr()
                capi.moe_decode_host(L["bank"], base, T, base + o_ids, base + o_w, hout[l].data_ptr(), io[l].data_ptr(),
                                     iob, self.ws.data_ptr(), self.ws_bytes, sp)

        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            launch(s.cuda_stream)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                launch(s.cuda_stream)
            for _ in range(warmup):
                g.replay()
            s.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(steps):
                g.replay()
                s.synchronize()
            e1.record(s)
            e1.synchronize()
        return e0.elapsed_time(e1) / steps, h2d, d2h

    def close(self):
        for L in self.layers:
            self.capi.moe_bank_destroy(L["bank"])
        self.layers = []


# ------------------------------------------------------------------ prompt path

# DRAM bytes of one k_layer_small launch (NVFP4 layer, T=1) from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum); valid only for the kernel
# source it was taken on.
# ncu DRAM bytes (read + write) of one headline k_layer_small launch, valid
# while the sources its code comes from are unchanged (one SHA-1 over them)
TRAFFIC = {"files": ["quantized_routed_expert_route_gb300/csrc/layer_small.cu",
                     "quantized_routed_expert_route_gb300/csrc/decode_common.cuh",
                     "quantized_routed_expert_route_gb300/csrc/formats.cuh",
                     "quantized_routed_expert_route_gb300/csrc/ptx.cuh"],
           "sha1": "95c2cc75a694dd2d6f465e355757b79704150548", "bytes": 21355264}


def traffic_bytes():
    import hashlib
    h = hashlib.sha1()
    for f in TRAFFIC["files"]:
        p = os.path.join(ROOT, f)
        if not os.path.exists(p):
            return None
        h.update(open(p, "rb").read())
    return TRAFFIC["bytes"] if h.hexdigest() == TRAFFIC["sha1"] else None


PREFILL = dict(H=2048, I=768, E=128, K=8, T=4096)


def prefill_flops(c):
    """Algorithmic FLOPs of one chunk: 2 per multiply-add of gate_up (2I x H)
    and down (H x I) for every routed row."""
    return 2.0 * c["T"] * c["K"] * (2 * c["I"] * c["H"] + c["H"] * c["I"])


def bench_prefill(dev, steps, warmup, mode, bf16_peak):
    """One NVFP4 layer (H=2048, I=768, E=128, top-8), a 4096-token chunk
    (32,768 routed rows) through moe_prefill_grouped; CUDA events around
    `steps` calls on one stream (weights 340 MB, beyond L2)."""
    import torch

    from quantized_routed_expert_route_gb300 import capi
    from synth import banks as S
    from synth import counter as C
    c = PREFILL
    H, I, E, K, T = c["H"], c["I"], c["E"], c["K"], c["T"]
    rb_gu, rb_dn = row_bytes(NVFP4, H), row_bytes(NVFP4, I)
    gu = torch.empty(E * 2 * I * rb_gu + 16, dtype=torch.uint8, device=dev)
    dn = torch.empty(E * H * rb_dn + 16, dtype=torch.uint8, device=dev)
    C.fill_bank_torch(gu[: E * 2 * I * rb_gu], 4001, NVFP4, H)
    C.fill_bank_torch(dn[: E * H * rb_dn], 4002, NVFP4, I)
    sb = torch.from_numpy(S.counter_scale_bank(4003, E, NVFP4, NVFP4)).to(dev)
    stream = torch.cuda.current_stream().cuda_stream
    geom = capi.moe_layer_geom(H, I, E, K, NVFP4, NVFP4)
    bank = capi.moe_bank_create(geom, gu.data_ptr(), E * 2 * I * rb_gu, dn.data_ptr(), E * H * rb_dn, sb.data_ptr(),
                                capi.MOE_SRC_DEVICE_BORROW, stream)
    ids, w = S.softmax_topk_routing(4004, T, E, K)
    x = torch.from_numpy(S.hidden_bf16(4005, T, H).view(np.int16)).to(dev)
    idsd, wd = torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev)
    out = torch.empty((T, H), dtype=torch.int16, device=dev)
    wsb = capi.moe_prefill_workspace_bytes(bank, T, mode)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)

    def call():
        capi.moe_prefill_grouped(bank, x.data_ptr(), T, idsd.data_ptr(), wd.data_ptr(), mode, out.data_ptr(),
                                 ws.data_ptr(), wsb, stream)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    err = capi.moe_get_error(ws.data_ptr(), wsb, stream)
    capi.moe_bank_destroy(bank)
    tflops = prefill_flops(c) / (ms / 1e3) / 1e12
    # algorithmic bytes: both banks once, x in and the bf16 output, ids and weights
    alg = E * 2 * I * rb_gu + E * H * rb_dn + 2 * T * H * 2 + 8 * T * K
    hbm_peak, _ = peaks()
    res = {"mode": {0: "W4A4", 1: "W4A8", 2: "FP16", 3: "W4A4 (fixed-order route sum)"}[mode], "ms_per_chunk": ms,
           "tok_per_s": T / (ms / 1e3),
           "tflops": tflops, "alg_bytes": alg, "hbm_gbs": alg / (ms / 1e3) / 1e9,
           "hbm_frac": alg / (ms / 1e3) / 1e9 / hbm_peak, "device_error_bits": err}
    if mode in (0, 3):
        # the FP4 peak: the measured bf16 peak times the nominal FP4 / BF16 ratio (13.5 / 2.25)
        res.update({"mma": "tcgen05 kind::mxf4nvf4 block-scaled FP4 (E2M1 x E2M1, UE4M3 per 16, fp32 accumulation), "
                           "operands by 2-D TMA",
                    "peak_tflops": bf16_peak * 6.0, "peak_kind": "measured bf16 x 6 (nominal FP4/BF16 ratio)",
                    "frac_of_fp4_peak": tflops / (bf16_peak * 6.0), "frac_of_nominal_fp4_peak": tflops / 13500.0,
                    "launches_per_chunk": 6})
    else:
        res.update({"mma": "tcgen05 kind::f16 (exact fp16 operands, fp32 accumulation)",
                    "frac_of_measured_bf16_peak": tflops / bf16_peak, "frac_of_nominal_fp4_peak": tflops / 13500.0,
                    "launches_per_chunk": 6})
    return res


def bench_linear(dev, steps, warmup, hbm_peak):
    """moe_linear on NVFP4 rows with per-row scales: 48 fused qkv projections
    of the headline layer shape (H=2048; q 4096 + k 512 + v 512 rows each,
    5.9 MB of rows per layer, 283 MB in all, beyond L2) as 48 launches
    replayed from one CUDA graph, and the same rows as one launch of
    245,760 rows.  T = 1 and 8; algorithmic bytes = rows + scales + x + out."""
    import torch

    from quantized_routed_expert_route_gb300 import capi
    from synth import banks as S
    from synth import counter as C
    NL, N, K = 48, 5120, 2048
    rb = row_bytes(NVFP4, K)
    rows = torch.empty(NL * N * rb + 16, dtype=torch.uint8, device=dev)
    C.fill_bank_torch(rows[: NL * N * rb], 5001, NVFP4, K)
    rs = torch.from_numpy(S.rng(5002).uniform(0.1, 2.0, size=NL * N).astype(np.float32)).to(dev)
    res = {"workload": "NVFP4 fused qkv rows, H=2048, N=5120 per layer, 48 layers (283 MB), per-row scales"}
    for T in (1, 8):
        x = torch.from_numpy(S.hidden_bf16(5003 + T, T, K).view(np.int16)).to(dev)
        out = torch.empty((NL, T, N), dtype=torch.int16, device=dev)
        big = torch.empty((T, NL * N), dtype=torch.int16, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        st = torch.cuda.Stream(device=dev)

        def layers(sp):
            for l in range(NL):
                capi.moe_linear(NVFP4, rows.data_ptr() + l * N * rb, N, K, rs.data_ptr() + 4 * l * N, x.data_ptr(),
                                T, out[l].data_ptr(), err.data_ptr(), sp)

        def one(sp):
            capi.moe_linear(NVFP4, rows.data_ptr(), NL * N, K, rs.data_ptr(), x.data_ptr(), T, big.data_ptr(),
                            err.data_ptr(), sp)

        with torch.cuda.stream(st):
            layers(st.cuda_stream)
            one(st.cuda_stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                layers(st.cuda_stream)
        torch.cuda.synchronize()
        row = {}
        for name, fn, nlaunch in (("48_layer_graph", lambda: g.replay(), NL),
                                  ("one_launch", lambda: one(st.cuda_stream), 1)):
            with torch.cuda.stream(st):
                for _ in range(warmup):
                    fn()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                for _ in range(steps):
                    fn()
                e1.record(st)
            e1.synchronize()
            ms = e0.elapsed_time(e1) / steps
            nbytes = NL * N * (rb + 4) + nlaunch * T * K * 2 + NL * N * T * 2   # rows + scales, x per launch, out
            gbs = nbytes / (ms / 1e3) / 1e9
            row[name] = {"us_per_step": ms * 1e3, "us_per_launch": ms * 1e3 / nlaunch, "hbm_gbs": gbs,
                         "frac": gbs / hbm_peak, "launches": nlaunch}
        row["device_error_bits"] = int(err.item())
        res[f"T={T}"] = row
        del g
    return res


def bench_cache(dev, tokens, hbm_peak):
    """Decode through the expert cache: four Laguna-shaped Q4_K layers
    (H=4096, I=768, E=256, top-10; 1.36 GB of compact rows each) live in
    pinned host memory; one pool of 160 slots (0.85 GB, 16 % of the 1,024
    experts) serves them.  A token runs the four layers in turn with Zipf
    routing: moe_cache_acquire (host LRU, copies of the missed experts) then
    moe_decode on the pool, all on one stream; timed with CUDA events over
    `tokens` tokens after a warm-up of 50."""
    import torch

    from quantized_routed_expert_route_gb300 import capi
    from synth import banks as S
    from synth import counter as C
    L, NL, NSLOTS = LAGUNA, 4, 160
    H, I, E, K = L["H"], L["I"], L["E"], L["K"]
    rb_gu, rb_dn = row_bytes(Q4_K, H), row_bytes(Q4_K, I)
    stream = torch.cuda.current_stream().cuda_stream
    host = []
    for l in range(NL):
        gu = torch.empty(E * 2 * I * rb_gu, dtype=torch.uint8, device=dev)
        dn = torch.empty(E * H * rb_dn, dtype=torch.uint8, device=dev)
        C.fill_bank_torch(gu, 7000 + 2 * l, Q4_K, H)
        C.fill_bank_torch(dn, 7001 + 2 * l, Q4_K, I)
        host.append((gu.cpu().pin_memory(), dn.cpu().pin_memory()))
        del gu, dn
    torch.cuda.empty_cache()
    cache = capi.moe_cache_create(capi.moe_layer_geom(H, I, NSLOTS, K, Q4_K, Q4_K), NSLOTS, stream)
    pool = capi.moe_cache_bank(cache)
    wsb = capi.moe_workspace_bytes(pool, 1)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    capi.moe_workspace_init(ws.data_ptr(), wsb, stream)
    n_all = 50 + tokens
    routes = [S.zipf_routing(7100 + l, n_all, E, K) for l in range(NL)]
    x = torch.from_numpy(S.hidden_bf16(7200, 1, H).view(np.int16)).to(dev)
    out = torch.empty((1, H), dtype=torch.int16, device=dev)
    sid = torch.empty((n_all, NL, K), dtype=torch.int32).pin_memory()
    sid_d = torch.empty((NL, K), dtype=torch.int32, device=dev)
    wts = [torch.from_numpy(w).to(dev) for _, w in routes]

    def token(t):
        for l in range(NL):
            ids = [int(v) for v in routes[l][0][t]]
            slots, _ = capi.moe_cache_acquire(cache, l, host[l][0].data_ptr(), host[l][1].data_ptr(), None, E, ids,
                                              stream)
            sid[t, l] = torch.tensor(slots, dtype=torch.int32)
            sid_d[l].copy_(sid[t, l], non_blocking=True)
            capi.moe_decode(pool, x.data_ptr(), 1, sid_d[l].data_ptr(), wts[l][t].data_ptr(), out.data_ptr(),
                            ws.data_ptr(), wsb, stream)

    for t in range(50):
        token(t)
    torch.cuda.synchronize()
    h0, m0, b0 = capi.moe_cache_stats(cache)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(50, n_all):
        token(t)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1)
    h1, m1, b1 = capi.moe_cache_stats(cache)
    err = capi.moe_get_error(ws.data_ptr(), wsb, stream)
    capi.moe_cache_destroy(cache)
    del host
    return {"workload": "4 Laguna-shaped Q4_K layers in pinned host memory (5.4 GB), 160-slot pool (0.85 GB), "
                        "T=1, Zipf(1.1) routing", "tokens": tokens,
            "tok_per_s": tokens / (ms / 1e3), "us_per_layer": ms * 1e3 / (tokens * NL),
            "hit_rate": (h1 - h0) / max(1, (h1 - h0) + (m1 - m0)), "misses_per_layer": (m1 - m0) / (tokens * NL),
            "h2d_gbs": (b1 - b0) / (ms / 1e3) / 1e9, "device_error_bits": err}


# ------------------------------------------------------------------ CPU oracle timing

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


_ORACLE_ROWS = {}


def _oracle_task(arg):
    """One pool task: `ntok` tokens of the headline layer through the oracle,
    in a process of its own (one BLAS thread); the routed experts' rows of the
    process's fixed routing are generated once per process, outside the
    timing.  Returns (tokens, oracle seconds)."""
    seed, ntok = arg
    from oracle import layer as OL
    from synth import banks as S
    from synth import counter as C
    c = CFG1
    geom = OL.Geometry(c["H"], c["I"], c["E"], c["K"], c["gu"], c["dn"])
    if seed not in _ORACLE_ROWS:
        ids, w = S.softmax_topk_routing(seed * 7, 1, c["E"], c["K"])
        gu, dn = {}, {}
        for e in (int(v) for v in ids.reshape(-1)):
            gu[e] = C.bank_bytes_np(seed * 1000, c["gu"], c["H"], e * 2 * c["I"], 2 * c["I"])
            dn[e] = C.bank_bytes_np(seed * 1000 + 1, c["dn"], c["I"], e * c["H"], c["H"])
        _ORACLE_ROWS[seed] = (ids, w, gu, dn, S.counter_scale_bank(seed * 1000, c["E"], c["gu"], c["dn"]), 0)
    ids, w, gu, dn, sb, n = _ORACLE_ROWS[seed]
    spent = 0.0
    for i in range(ntok):
        x = S.hidden_bf16(seed * 131 + n + i, 1, c["H"])
        t0 = time.perf_counter()
        OL.moe_layer(geom, gu, dn, sb, x, ids, w)
        spent += time.perf_counter() - t0
    _ORACLE_ROWS[seed] = (ids, w, gu, dn, sb, n + ntok)
    return ntok, spent


class OraclePool:
    """A spawn pool of oracle processes, one per host core, each with one BLAS
    thread and no GPU (started before any CUDA call of this process)."""

    def __init__(self, n: int):
        import multiprocessing as mp
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
        saved = os.environ.get("CUDA_VISIBLE_DEVICES")
        os.environ["CUDA_VISIBLE_DEVICES"] = ""
        self.n = n
        self.pool = mp.get_context("spawn").Pool(n)
        if saved is None:
            del os.environ["CUDA_VISIBLE_DEVICES"]
        else:
            os.environ["CUDA_VISIBLE_DEVICES"] = saved

    def rate(self, ntok: int, seed0: int, procs: int | None = None) -> tuple[float, int]:
        """Summed throughput (tokens / oracle second, over the processes) of
        `ntok` tokens in each of `procs` processes at once."""
        k = self.n if procs is None else procs
        res = self.pool.map(_oracle_task, [(seed0 + i, ntok) for i in range(k)], chunksize=1)
        return sum(t / s for t, s in res), sum(t for t, _ in res)

    def close(self):
        self.pool.terminate()
        self.pool.join()


def run_cpu_baseline(pool: "OraclePool", seconds: float) -> dict:
    """The oracle on the host cores: one process alone, then every process at
    once (one per core, tokens split across them, throughput summed), each
    for about `seconds` of oracle time."""
    try:
        pool.rate(1, 0, procs=pool.n)                        # rows generated, imports warm
        one, t1 = pool.rate(max(1, int(seconds * 1.5)), 0, procs=1)
        many, tn = pool.rate(max(1, int(seconds * 1.5)), 0)
    except Exception as e:   # noqa: BLE001 (reported in the line, the bench goes on)
        return {"value": None, "unit": "layer-tok/s", "cores": 1, "kind": "oracle", "sample": f"failed: {e}"}
    return {"value": many, "unit": "layer-tok/s", "cores": pool.n, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{pool.n} oracle processes at once (one per core, one BLAS thread each), {tn} tokens of one "
                      f"NVFP4 layer (H=2048, I=768, E=128, top-8) in all, numpy fp64; throughput summed over the "
                      f"processes",
            "single_core": {"value": one, "cores": 1, "sample": f"{t1} tokens in one process"}}


# ------------------------------------------------------------------ profiling driver

def summary_of(line: dict) -> dict:
    """A compact digest of the line (rounded): the headline, the Laguna stack
    sweep, the other-type layers, the prompt chunk, the dense linear, the
    expert cache and the CPU baseline."""
    ex = line.get("extra", {})
    r3 = lambda v: None if v is None else float(f"{v:.3g}")   # noqa: E731
    s = {"layer_us_T1": r3(ex.get("per_layer_us")), "hbm_frac_T1": r3(line["roofline"]["frac"]),
         "layer_us_T8": r3(ex.get("t8", {}).get("per_layer_us"))}
    if "laguna_47_layer_stack" in ex:
        s["laguna_stack"] = {k: {"tok_s": r3(v["stack_tok_per_s"]), "hbm_frac": r3(v["frac"])}
                             for k, v in ex["laguna_47_layer_stack"].items()}
    if "gguf_types_24_layer_stack" in ex:
        s["types_layer_us_T1_T8"] = {k: [r3(v["T=1"]["per_layer_us"]), r3(v["T=8"]["per_layer_us"])]
                                     for k, v in ex["gguf_types_24_layer_stack"].items() if k != "workload"}
    if "prefill_4096_token_chunk" in ex:
        pf = ex["prefill_4096_token_chunk"]
        s["prefill_chunk_ms"] = {m: r3(pf[m]["ms_per_chunk"]) for m in ("w4a4", "w4a4_fixed", "w4a8", "fp16") if m in pf}
        s["prefill_tflops"] = {m: r3(pf[m]["tflops"]) for m in ("w4a4", "w4a4_fixed", "w4a8", "fp16") if m in pf}
        if "w4a4" in pf:
            s["prefill_w4a4_frac_nominal_fp4"] = r3(pf["w4a4"].get("frac_of_nominal_fp4_peak"))
    if "dense_linear_nvfp4" in ex:
        dl = ex["dense_linear_nvfp4"]
        s["linear_one_launch_hbm_frac"] = {k: r3(dl[k]["one_launch"]["frac"]) for k in ("T=1", "T=8") if k in dl}
    if "expert_cache" in ex:
        s["cache_tok_s"] = r3(ex["expert_cache"].get("tok_per_s"))
    cpu = line.get("cpu_baseline") or {}
    s["cpu_oracle"] = {"value": r3(cpu.get("value")), "cores": cpu.get("cores"),
                       "single_core": r3((cpu.get("single_core") or {}).get("value"))}
    return s


def profile_layer(a):
    """Eager decode passes of one layer for a profiler: the NVFP4 layer
    (H=2048, I=768, E=128, top-8) or the same shape with Q4_K+Q6_K, Q6_K or
    Q4_0 rows, or a Laguna-shaped Q4_K / BF16 layer
    (H=4096, I=768, E=256, top-10, Zipf routing), a stack of --layers banks."""
    import torch
    dev = "cuda:0"
    other = {"q4_k_m": (Q4_K, Q6_K), "q6_k": (Q6_K, Q6_K), "q4_0": (Q4_0, Q4_0)}
    if a.profile_layer == "nvfp4" or a.profile_layer in other:
        c = CFG1
        pair = other.get(a.profile_layer, (c["gu"], c["dn"]))
        st = Stack([pair] * a.layers, c["H"], c["I"], c["E"], c["K"], 1, dev)
        st.prepare(a.T, "softmax", 1)
    else:
        t = Q4_K if a.profile_layer == "q4_k" else BF16
        L = LAGUNA
        st = Stack([(t, t)] * a.layers, L["H"], L["I"], a.experts or L["E"], L["K"], 3, dev)
        st.prepare(a.T, "zipf", 3 + a.T)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(a.steps):
        st.launch_all(s)
    torch.cuda.synchronize()
    st.close()
    print(json.dumps({"profile_layer": a.profile_layer, "T": a.T, "layers": a.layers, "steps": a.steps}))


def profile_linear(a):
    """Eager one-launch dense NVFP4 linears (the bench's 283 MB of rows) for a profiler."""
    import torch

    from quantized_routed_expert_route_gb300 import capi
    from synth import counter as C
    dev = "cuda:0"
    N, K = 48 * 5120, 2048
    rb = row_bytes(NVFP4, K)
    rows = torch.empty(N * rb + 16, dtype=torch.uint8, device=dev)
    C.fill_bank_torch(rows[: N * rb], 5001, NVFP4, K)
    rs = torch.ones(N, dtype=torch.float32, device=dev)
    x = torch.zeros((a.T, K), dtype=torch.int16, device=dev)
    out = torch.empty((a.T, N), dtype=torch.int16, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(a.steps):
        capi.moe_linear(NVFP4, rows.data_ptr(), N, K, rs.data_ptr(), x.data_ptr(), a.T, out.data_ptr(), None, s)
    torch.cuda.synchronize()
    print(json.dumps({"profile_linear": True, "T": a.T, "steps": a.steps}))


# ------------------------------------------------------------------ main

def job_throughput(ms_local, units_per_rank, world, device):
    """Whole-job throughput of independent replicas: the units every rank
    processed, over the slowest rank's time (max over ranks).  Returns
    (units per second, max ms)."""
    t_max = ms_local
    if world > 1:
        import torch
        tt = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        t_max = float(tt.item())
    return units_per_rank * world / (t_max / 1e3), t_max


def dist_setup(n):
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return dist.get_rank(), dist.get_world_size(), local
    return 0, 1, 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=48)
    ap.add_argument("--no-stack", action="store_true", help="skip the 47-layer Laguna sweep")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prompt-path chunk")
    ap.add_argument("--no-types", action="store_true", help="skip the per-GGUF-type layer stacks")
    ap.add_argument("--no-linear", action="store_true", help="skip the dense NVFP4 linear")
    ap.add_argument("--no-cache", action="store_true", help="skip the expert-cache leg")
    ap.add_argument("--profile-linear", action="store_true",
                    help="run --steps one-launch dense NVFP4 linears (245,760 x 2048, T=--T) for ncu")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--profile-layer", choices=["nvfp4", "q4_k", "bf16", "q4_k_m", "q6_k", "q4_0"], default=None,
                    help="run --steps eager decode passes of one layer type (for ncu), print nothing else")
    ap.add_argument("--T", type=int, default=1)
    ap.add_argument("--experts", type=int, default=0,
                    help="with --profile-layer q4_k/bf16: experts per layer (default 256), to shrink a capture")
    ap.add_argument("--profile-prefill", choices=["w4a4", "w4a4_fixed", "w4a8", "fp16"], default=None,
                    help="run --steps prompt-path chunks (for ncu), print nothing else")
    a = ap.parse_args()

    if a.profile_layer:
        profile_layer(a)
        return
    if a.profile_prefill:
        import torch
        r = bench_prefill("cuda:0", a.steps, 1, {"w4a4": 0, "w4a8": 1, "fp16": 2, "w4a4_fixed": 3}[a.profile_prefill],
                          bf16_peak()[0])
        print(json.dumps(r))
        return

    if a.profile_linear:
        profile_linear(a)
        return

    workload = (f"qwen3-30b-a3b-shaped nvfp4 routed-expert decode layer (H=2048, I=768, E=128, top-8, T=1), "
                f"{a.layers} distinct resident layer banks per step")
    # both arms print the same metric and config
    metric = "routed-expert decode throughput (tokens x layers / s); achieved HBM GB/s vs peak"

    def config(world):
        return {"workload": workload, "T": 1, "layers_per_step": a.layers,
                "l2": "inputs larger than L2 (1 GB of expert rows per step, 16 GB resident)",
                "parallelism": f"replicas x{world}"}

    if a.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        pool = OraclePool(os.cpu_count() or 1)
        pool.rate(1, 1000, procs=pool.n)   # rows generated, imports warm (outside the steps)
        vals = []
        for i in range(a.warmup + a.steps):
            v, _ = pool.rate(1, 1000)
            if i >= a.warmup:
                vals.append(v)
        pool.close()
        v = float(np.mean(vals))
        print(json.dumps({
            "impl": "reference", "metric": metric, "value": v, "unit": "layer-tok/s",
            "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup, "higher_is_better": True,
            "dtype": "f64", "data": "synthetic", "config": config(a.gpus),
            "cpu_baseline": {"kind": "oracle", "cores": pool.n, "value": v, "cpu_model": cpu_model(),
                             "sample": f"per step: one token of one NVFP4 layer in each of {pool.n} oracle "
                                       f"processes at once (one per core); throughput summed"},
            "e2e": {"value": v, "unit": "layer-tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return

    # the oracle's process pool starts before any CUDA call of this process
    rank0 = int(os.environ.get("RANK", "0")) == 0
    pool = OraclePool(os.cpu_count() or 1) if (rank0 and a.cpu_seconds > 0) else None

    import torch
    rank, world, local = dist_setup(a.gpus)
    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    hbm_peak, peak_kind = peaks()

    # headline: NVFP4 layer stack, T=1
    c = CFG1
    st = Stack([(c["gu"], c["dn"])] * a.layers, c["H"], c["I"], c["E"], c["K"], 1, dev)
    st.prepare(1, "softmax", 1)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = st.time_replays(a.steps, a.warmup)
    value, t_max = job_throughput(ms, a.layers * 1, world, dev)   # layer-tokens per step per rank
    units = a.layers * 1 * world                                   # whole job
    per_pass_ms = ms / a.layers
    achieved = st.bytes_per_step / a.layers / (per_pass_ms / 1e3) / 1e9
    launches = st.launches_per_step * a.steps
    e2e_ms, h2d, d2h = st.time_e2e(max(10, a.steps // 4), a.warmup)
    e2e_val = units / (e2e_ms / 1e3)
    extra = {"per_layer_us": per_pass_ms * 1e3, "bytes_per_layer": st.bytes_per_step / a.layers,
             "unique_experts_per_layer": float(np.mean(st.unique_per_layer))}

    # the same NVFP4 layer stack at T=8
    st.prepare(8, "softmax", 2)
    ms8 = st.time_replays(max(10, a.steps // 2), a.warmup)
    extra["t8"] = {"layer_tok_per_s": a.layers * 8 / (ms8 / 1e3), "per_layer_us": ms8 / a.layers * 1e3,
                   "hbm_gbs": st.bytes_per_step / (ms8 / 1e3) / 1e9}
    st.close()
    del st
    torch.cuda.empty_cache()

    if not a.no_stack:
        L = LAGUNA
        types = [(BF16, BF16) if l % 6 == 0 else (Q4_K, Q4_K) for l in range(47)]
        sweep = {}
        st = Stack(types, L["H"], L["I"], L["E"], L["K"], 3, dev)
        for T in (1, 4, 16, 64):
            st.prepare(T, "zipf", 3 + T)
            msT = st.time_replays(max(5, min(20, a.steps // 5)), a.warmup)
            sweep[f"T={T}"] = {"stack_tok_per_s": T / (msT / 1e3), "ms_per_stack": msT,
                               "hbm_gbs": st.bytes_per_step / (msT / 1e3) / 1e9,
                               "frac": st.bytes_per_step / (msT / 1e3) / 1e9 / hbm_peak,
                               "gb_per_step": st.bytes_per_step / 1e9}
        st.close()
        del st
        torch.cuda.empty_cache()
        extra["laguna_47_layer_stack"] = sweep

    if not a.no_types:
        c = CFG1
        types = {}
        for gu_t, dn_t in TYPE_PAIRS:
            st = Stack([(gu_t, dn_t)] * 24, c["H"], c["I"], c["E"], c["K"], 5, dev)
            row = {}
            for T in (1, 8):
                st.prepare(T, "softmax", 11 + T)
                msT = st.time_replays(max(10, min(100, a.steps // 4)), a.warmup)
                gbs = st.bytes_per_step / (msT / 1e3) / 1e9
                row[f"T={T}"] = {"per_layer_us": msT / 24 * 1e3, "layer_tok_per_s": 24 * T / (msT / 1e3),
                                 "hbm_gbs": gbs, "frac": gbs / hbm_peak,
                                 "launches_per_layer": st.launches_per_step / 24}
            st.close()
            del st
            torch.cuda.empty_cache()
            types[f"{TYPE_NAMES[gu_t]}+{TYPE_NAMES[dn_t]}"] = row
        extra["gguf_types_24_layer_stack"] = {
            "workload": "H=2048 I=768 E=128 top-8, softmax routing, 24 resident layer banks per step", **types}

    if not a.no_linear:
        extra["dense_linear_nvfp4"] = bench_linear(dev, max(10, min(100, a.steps // 4)), a.warmup, hbm_peak)
        torch.cuda.empty_cache()

    if not a.no_cache:
        extra["expert_cache"] = bench_cache(dev, max(50, min(400, a.steps)), hbm_peak)
        torch.cuda.empty_cache()

    if not a.no_prefill:
        pk, pk_kind = bf16_peak()
        extra["prefill_4096_token_chunk"] = {
            "workload": "nvfp4 layer H=2048 I=768 E=128 top-8, 4096 tokens (32768 routed rows)",
            "peak_tflops": pk, "peak_kind": pk_kind, "gflop_per_chunk": prefill_flops(PREFILL) / 1e9,
            "w4a4": bench_prefill(dev, max(3, min(20, a.steps // 20)), a.warmup, 0, pk),
            "w4a4_fixed": bench_prefill(dev, max(3, min(20, a.steps // 20)), a.warmup, 3, pk),
            "w4a8": bench_prefill(dev, max(3, min(20, a.steps // 20)), a.warmup, 1, pk),
            "fp16": bench_prefill(dev, max(3, min(20, a.steps // 20)), a.warmup, 2, pk)}
        torch.cuda.empty_cache()

    cpu = run_cpu_baseline(pool, a.cpu_seconds / 2) if pool is not None else None
    if pool is not None:
        pool.close()
    if rank == 0:
        line = {
            "metric": metric,
            "value": value, "unit": "layer-tok/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": t_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "nvfp4 weights x q8_1 activations, int32 block dots, fp32 epilogue, bf16 out",
            "data": "synthetic (counter-based banks, seeded routings)",
            "config": config(world),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": traffic_bytes(), "peak_kind": peak_kind,
                         "kernel": "k_layer_small (one fused launch per moe_decode pass at T=1)"},
            "clocks": clk.summary(),
            "e2e": {"value": e2e_val, "unit": "layer-tok/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "cpu_baseline": cpu,
            "extra": extra,
        }
        line["summary"] = summary_of(line)   # last, so a tail of the output keeps it
        print(json.dumps(line))
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
