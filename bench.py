"""Benchmark of the W4A8 packed-linear path on GB300 (one JSON line on stdout).

Workloads (synthetic, seeded; shapes of Qwen2.5-7B linears and DiT blocks):
  decode   (default) one step = for M in {1, 4, 16}: per-token int8 quantization
           of the four linear inputs + the seven W4A8 linears q,k,v,o,gate,up,down.
           Layer copies rotate so the weights streamed per step exceed L2.
  prefill  one step = for M in {512, 2048, 4096}: the same seven linears plus the
           untied quantized output head (K=3584, N=152064).
  model    one step = the full linear pass: 28 layers x 7 = 196 W4A8 linears +
           head at one M (--m, default 1), independent weights per layer.
  dit      one step = W4A16 and W8A16 on K=3072,N in {3072,12288} and
           K=12288,N=3072 at M in {1, 16, 4096}.
  tiny     M=16, K=512, N=256 (the oracle-sized case).
  linear   one W4A8 linear of --k/--n at --m tokens (used for profiling captures).

value = algorithmic bytes (decode, dit-weight-only at M<=16) or algorithmic
integer ops (prefill) per second over K timed steps, inputs resident in HBM.
e2e   = the same metric through the public API with the step's activations
        copied from pinned host memory and its outputs copied back each step.
--impl reference times the CPU oracle (the reference arm of this build) on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A8 GEMM TOPS and HBM GB/s (% of roofline) on 7B-shaped linears, M=1–4096"
SHAPES_7B = [("q", 3584, 3584), ("k", 3584, 512), ("v", 3584, 512), ("o", 3584, 3584),
             ("gate", 3584, 18944), ("up", 3584, 18944), ("down", 18944, 3584)]
HEAD = ("head", 3584, 152064)
INPUT_OF = {"q": "attn", "k": "attn", "v": "attn", "o": "o", "gate": "mlp", "up": "mlp",
            "down": "down"}
INPUT_K = {"attn": 3584, "o": 3584, "mlp": 3584, "down": 18944, "head": 3584}
FUSED = {"qkv": ["q", "k", "v"], "gate_up": ["gate", "up"]}
INPUT_OF.update({"qkv": "attn", "gate_up": "mlp"})


def fuse_shapes(shapes):
    """Sibling linears sharing an input as one GEMM (weights concatenated along N)."""
    out, seen = [], set()
    for (nm, K, N) in shapes:
        group = next((f for f, parts in FUSED.items() if nm in parts), None)
        if group is None:
            out.append((nm, K, N))
        elif group not in seen:
            seen.add(group)
            out.append((group, K, sum(n for (x, _, n) in shapes if x in FUSED[group])))
    return out


def pack_linear(eg, synth, t, torch, config, layer, nm, N, K):
    """Pack one linear (or a fused sibling group, each part drawn from its own
    seed so the data equal the unfused linears')."""
    import numpy as np
    parts = FUSED.get(nm, [nm])
    ws = [synth.w4_weights(config, layer, synth.LINEARS.get(p, 0),
                           {"q": 3584, "k": 512, "v": 512, "gate": 18944, "up": 18944}.get(p, N)
                           if len(parts) > 1 else N, K) for p in parts]
    w_q = np.concatenate([w.w_q for w in ws])
    s = np.concatenate([w.scale_f16 for w in ws])
    z = np.concatenate([w.zero for w in ws])
    assert w_q.shape == (N, K)
    return eg.pack_w4(t(w_q), t(s, torch.float16), t(z))
G128 = 128


def w4a8_bytes(M, N, K):
    G = K // G128
    return N * K // 2 + 2 * N * G + N * G // 2 + M * K + 4 * M + 4 * M * G + 2 * M * N


def quant_bytes(M, K):
    return 2 * M * K + M * K + 4 * M + 4 * M * (K // G128)


def w4a16_bytes(M, N, K):
    G = K // G128
    return N * K // 2 + 2 * N * G + N * G // 2 + 2 * M * K + 2 * M * N


def w8a16_bytes(M, N, K):
    return N * K + 2 * N + 2 * M * K + 2 * M * N


def w8a8_bytes(M, N, K):
    return N * K + 2 * N + M * K + 4 * M + 2 * M * N


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_sources_hash() -> str:
    """sha256 over the CUDA sources and the public header (names and bytes)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "w4a8_quantized_gemm_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc)
                   if f.endswith((".cu", ".cuh", ".h")))
    files.append(os.path.join(ROOT, "include", "egopq.h"))
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def config_key(args) -> str:
    return (f"{args.workload}|path={args.path}|fused={int(args.fused)}|api={args.api}|"
            f"m={args.m}|k={args.k}|n={args.n}|variant={args.variant}")


def measured_traffic(args, kernel_label: str):
    """DRAM bytes per launch of `kernel_label` on this configuration, from the
    ncu capture summarised in profiles/dram_traffic.txt, or None when there is
    none or the kernels changed since it was taken (source hash mismatch)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want_hash, key = None, config_key(args)
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line.startswith("sources_sha256="):
                want_hash = line.split("=", 1)[1]
            elif line.startswith("config=") and want_hash is not None:
                fields = dict(kv.split("=", 1) for kv in line.split("\t"))
                if fields["config"] == key and fields["kernel"] == kernel_label:
                    if want_hash != kernel_sources_hash():
                        return None
                    return float(fields["bytes_per_launch"])
    return None


# ------------------------------------------------------------------ clocks ----

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(value: float, device=None) -> float:
    """Replicas only: the one cross-rank step is this timing reduction (MAX),
    followed by a barrier. Works on NCCL (device tensor) and gloo (CPU)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


# --------------------------------------------------------------- workloads ----

class Workload:
    """A list of launches per step ("ops"), built once; inputs resident on device."""

    def __init__(self, name, dev, copies=None, m=1, lin=(3584, 3584), path=0, variant="w4a8",
                 fused=False, api="gemm"):
        import torch

        import synth
        import w4a8_quantized_gemm_gb300 as eg
        self.torch, self.eg, self.dev, self.name, self.path = torch, eg, dev, name, path
        self.api, self._ws = api, {}
        self.twin_specs = {}
        self.steps_ops = []   # per layer copy: list of (kind, callable-args)
        self.ops_meta = []    # (kind, M, N, K, bytes, ops)
        self.inputs = []      # per copy: list of device tensors fed from host in e2e
        self.outputs = []
        t = lambda a, dt=None: _to_dev(torch, a, dev, dt)
        if name == "linear" and variant != "w4a8":  # weight-only single linear
            name = self.name = "dit"
        if name in ("decode", "prefill", "tiny", "linear"):
            if name == "decode":
                ms, shapes, n_copies = [1, 4, 16], SHAPES_7B, copies or 4
            elif name == "prefill":
                ms, shapes, n_copies = [512, 2048, 4096], SHAPES_7B + [HEAD], copies or 1
            elif name == "linear":
                ms, shapes, n_copies = [m], [("q", lin[0], lin[1])], copies or 1
            else:
                ms, shapes, n_copies = [16], [("q", 512, 256)], copies or 1
            if fused and name in ("decode", "prefill"):
                shapes = fuse_shapes(shapes)
            self.layers = []
            for c in range(n_copies):
                packs = {}
                for (nm, K, N) in shapes:
                    packs[nm] = pack_linear(eg, synth, t, torch, 1, c, nm, N, K)
                self.layers.append(packs)
            torch.cuda.synchronize()
            self.ms = ms
            self.shapes = shapes
            self.acts = {}
            for M in ms:
                for inp in sorted(set(INPUT_OF.get(nm, "head") for nm, _, _ in shapes)):
                    K = {"tiny": 512, "linear": shapes[0][1]}.get(name, INPUT_K.get(inp))
                    x = synth.activations(1, 0, {"attn": 0, "o": 3, "mlp": 4, "down": 6,
                                                 "head": 7}[inp], M, K)
                    xd = t(x, torch.bfloat16)
                    a = eg.QuantAct(torch.empty((M, K), dtype=torch.int8, device=dev),
                                    torch.empty((M,), dtype=torch.float32, device=dev),
                                    torch.empty((M, K // G128), dtype=torch.int32, device=dev),
                                    eg.tc_operand(M, K, dev))
                    self.acts[(M, inp)] = (x, xd, a)
            self.ys = {(M, nm): torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                       for M in ms for (nm, K, N) in shapes}
        elif name == "model":
            self.ms = [m]
            self.shapes = fuse_shapes(SHAPES_7B) if fused else SHAPES_7B
            self.layers = []
            for layer in range(28):
                packs = {}
                for (nm, K, N) in self.shapes:
                    packs[nm] = pack_linear(eg, synth, t, torch, 3, layer, nm, N, K)
                self.layers.append(packs)
            wh = synth.w4_weights(3, 0, synth.LINEARS["head"], HEAD[2], HEAD[1])
            self.head = eg.pack_w4(t(wh.w_q), t(wh.scale_f16, torch.float16), t(wh.zero))
            torch.cuda.synchronize()
            self.acts = {}
            for inp in ["attn", "o", "mlp", "down", "head"]:
                K = INPUT_K[inp]
                x = synth.activations(3, 0, {"attn": 0, "o": 3, "mlp": 4, "down": 6,
                                             "head": 7}[inp], m, K)
                a = eg.QuantAct(torch.empty((m, K), dtype=torch.int8, device=dev),
                                torch.empty((m,), dtype=torch.float32, device=dev),
                                torch.empty((m, K // G128), dtype=torch.int32, device=dev),
                                eg.tc_operand(m, K, dev))
                self.acts[(m, inp)] = (x, t(x, torch.bfloat16), a)
            self.ys = {(m, nm): torch.empty((m, N), dtype=torch.bfloat16, device=dev)
                       for (nm, K, N) in self.shapes + [HEAD]}
        if name == "dit":
            self.ms = [1, 16, 4096] if variant == "w4a8" else [m]
            self.dit_shapes = ([(3072, 3072), (3072, 12288), (12288, 3072)]
                               if variant == "w4a8" else [tuple(lin)])
            self.dit_variants = {"w4a8": ("w4", "w8"), "w4a16": ("w4",), "w8a16": ("w8",),
                                 "w8a8": ("w8a8",)}[variant]
            self.dit_w = {}
            for (K, N) in self.dit_shapes:
                w = synth.w4_weights(4, 0, 0, N, K)
                w8, s8 = synth.w8_weights(4, 0, 0, N, K)
                self.dit_w[(K, N)] = (eg.pack_w4(t(w.w_q), t(w.scale_f16, torch.float16),
                                                 t(w.zero)), t(w8), t(s8, torch.float16))
            self.acts = {}
            for M in self.ms:
                for K in sorted(set(k for k, _ in self.dit_shapes)):
                    x = synth.activations(4, 0, 0, M, K, outliers=False)
                    self.acts[(M, K)] = (x, t(x, torch.bfloat16))
            # W8A8: per-token int8 codes (the tensor-core operand form only
            # where that path runs)
            self.qacts = {(M, K): eg.QuantAct(
                torch.empty((M, K), dtype=torch.int8, device=dev),
                torch.empty((M,), dtype=torch.float32, device=dev),
                torch.empty((M, K // G128), dtype=torch.int32, device=dev),
                eg.tc_operand(M, K, dev) if M > eg.TC_FP8_MAX_M else None)
                for (M, K) in self.acts} if "w8a8" in self.dit_variants else {}
            self.ys = {(M, K, N, v): torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                       for M in self.ms for (K, N) in self.dit_shapes for v in self.dit_variants}
            self.layers = [None]
        elif name not in ("decode", "prefill", "tiny", "linear", "model"):
            raise ValueError(name)
        self.n_copies = 1 if name == "model" else len(self.layers)
        self._pack_io()

    def _pack_io(self):
        """Place every bf16 activation input in one device buffer and every
        output in another (views keep their shapes; sizes are multiples of 256
        bytes, so each view stays 16-byte aligned), so that the end-to-end leg
        moves each step's inputs and outputs with one copy each way."""
        torch = self.torch

        def pack(tensors):
            total = sum(t.numel() for t in tensors)
            buf = torch.empty((total,), dtype=torch.bfloat16, device=self.dev)
            views, off = [], 0
            for t in tensors:
                v = buf[off:off + t.numel()].view(t.shape)
                v.copy_(t)
                views.append(v)
                off += t.numel()
            return buf, views

        keys = list(self.acts.keys())
        self.x_all, xs = pack([self.acts[k][1] for k in keys])
        for k, v in zip(keys, xs):
            self.acts[k] = (self.acts[k][0], v) + tuple(self.acts[k][2:])
        ykeys = list(self.ys.keys())
        self.y_all, yv = pack([self.ys[k] for k in ykeys])
        self.ys = dict(zip(ykeys, yv))

    # one step's launches, as (label, kind, M, N, K, bytes, ops, fn)
    def step_ops(self, copy: int):
        eg, ops = self.eg, []
        # the same products on dense bf16 weights, for the twin leg:
        # (label, M, N, K, bf16 activations, packed int4 weight, output)
        twins = self.twin_specs.setdefault(copy, [])
        twins.clear()
        if self.name in ("decode", "prefill", "tiny", "linear", "model"):
            layers = [self.layers[copy]] if self.name != "model" else self.layers
            for M in self.ms:
                for li, packs in enumerate(layers):
                    done = set()
                    for (nm, K, N) in self.shapes:
                        inp = INPUT_OF.get(nm, "head") if self.name not in ("tiny", "linear") \
                            else "attn"
                        x, xd, a = self.acts[(M, inp)]
                        if self.api == "linear":
                            # same algorithmic bytes as the two-call step: the
                            # first linear of each input carries its quantization
                            qb = 0 if inp in done else quant_bytes(M, K)
                            done.add(inp)
                            y = self.ys[(M, nm)]
                            ws = self.workspace(M, K)
                            ops.append((f"{nm} M={M}", "w4a8", M, N, K,
                                        w4a8_bytes(M, N, K) + qb, 2 * M * N * K,
                                        (lambda xd=xd, p=packs[nm], N=N, y=y, ws=ws:
                                         eg.w4a8_linear(xd, p, N, out=y, workspace=ws,
                                                        path=self.path))))
                            continue
                        if inp not in done:
                            done.add(inp)
                            ops.append((f"quant {inp} M={M}", "quant", M, 0, K,
                                        quant_bytes(M, K), 0,
                                        (lambda xd=xd, a=a: eg.quant_act(xd, out=a))))
                        y = self.ys[(M, nm)]
                        twins.append((f"{nm} M={M}", M, N, K, xd, packs[nm], y))
                        ops.append((f"{nm} M={M}", "w4a8", M, N, K, w4a8_bytes(M, N, K),
                                    2 * M * N * K,
                                    (lambda a=a, p=packs[nm], N=N, K=K, y=y:
                                     eg.w4a8_gemm(a, p, N, K, out=y, path=self.path))))
                if self.name == "model":
                    x, xd, a = self.acts[(M, "head")]
                    K, N = HEAD[1], HEAD[2]
                    ops.append((f"quant head M={M}", "quant", M, 0, K, quant_bytes(M, K), 0,
                                (lambda xd=xd, a=a: eg.quant_act(xd, out=a))))
                    y = self.ys[(M, "head")]
                    twins.append((f"head M={M}", M, N, K, xd, self.head, y))
                    ops.append((f"head M={M}", "w4a8", M, N, K, w4a8_bytes(M, N, K),
                                2 * M * N * K,
                                (lambda a=a, p=self.head, N=N, K=K, y=y:
                                 eg.w4a8_gemm(a, p, N, K, out=y, path=self.path))))
        else:
            quantized = set()
            for M in self.ms:
                for (K, N) in self.dit_shapes:
                    x, xd = self.acts[(M, K)]
                    p4, w8, s8 = self.dit_w[(K, N)]
                    if "w8a8" in self.dit_variants:
                        a = self.qacts[(M, K)]
                        if (M, K) not in quantized:
                            quantized.add((M, K))
                            ops.append((f"quant K={K} M={M}", "quant", M, 0, K,
                                        quant_bytes(M, K), 0,
                                        (lambda xd=xd, a=a: eg.quant_act(xd, out=a))))
                        y = self.ys[(M, K, N, "w8a8")]
                        ops.append((f"w8a8 K={K} N={N} M={M}", "w8a8", M, N, K,
                                    w8a8_bytes(M, N, K), 2 * M * N * K,
                                    (lambda a=a, w8=w8, s8=s8, y=y:
                                     eg.w8a8_gemm(a, w8, s8, out=y, path=self.path))))
                    if "w4" in self.dit_variants:
                        y4 = self.ys[(M, K, N, "w4")]
                        twins.append((f"K={K} N={N} M={M}", M, N, K, xd, p4, y4))
                        ops.append((f"w4a16 K={K} N={N} M={M}", "w4a16", M, N, K,
                                    w4a16_bytes(M, N, K), 2 * M * N * K,
                                    (lambda xd=xd, p=p4, N=N, K=K, y=y4:
                                     eg.w4a16_gemm(xd, p, N, K, out=y, path=self.path))))
                    if "w8" in self.dit_variants:
                        y8 = self.ys[(M, K, N, "w8")]
                        ops.append((f"w8a16 K={K} N={N} M={M}", "w8a16", M, N, K,
                                    w8a16_bytes(M, N, K), 2 * M * N * K,
                                    (lambda xd=xd, w8=w8, s8=s8, y=y8:
                                     eg.w8a16_gemm(xd, w8, s8, out=y, path=self.path))))
        return ops

    def workspace(self, M, K):
        """Device workspace of the one-call linear, shared by every call of one
        (M, K) (calls are ordered on one stream)."""
        need = self.eg.w4a8_linear_workspace_bytes(M, K, self.path)
        if not need:
            return None
        key = (M, K)
        if key not in self._ws:
            self._ws[key] = self.torch.empty(need, dtype=self.torch.uint8, device=self.dev)
        return self._ws[key]

    def host_io(self):
        """([(pinned host inputs, device inputs)], [(device outputs, pinned host
        outputs)]) for the end-to-end leg: one buffer each way (see _pack_io)."""
        torch = self.torch
        x_host = torch.empty(self.x_all.shape, dtype=self.x_all.dtype).pin_memory()
        x_host.copy_(self.x_all.cpu())
        y_host = torch.empty(self.y_all.shape, dtype=self.y_all.dtype).pin_memory()
        return [(x_host, self.x_all)], [(self.y_all, y_host)]


def _to_dev(torch, a, dev, dt=None):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a).to(dev)
    return t.view(dt) if dt is not None else t


def kernel_label(eg, kind, M, path):
    if kind == "quant":
        return "quant_act_kernel"
    if kind == "w4a8":
        gemv = path == eg.PATH_GEMV or (path == eg.PATH_AUTO and M <= eg.GEMV_AUTO_MAX_M)
        return "gemv_w4_kernel (W4A8)" if gemv else "tc_gemm_kernel (W4A8)"
    if kind == "w8a8":
        gemv = path == eg.PATH_GEMV or (path == eg.PATH_AUTO and M <= eg.TC_FP8_MAX_M)
        return "gemv_w8a8_kernel (W8A8)" if gemv else "tc_gemm_kernel (W8A8)"
    if path == eg.PATH_GEMV:  # weight-only GEMVs run only when forced
        return "gemv_w8_kernel (W8A16)" if kind == "w8a16" else "gemv_w4_kernel (W4A16)"
    return f"tc_gemm_kernel ({kind.upper()})"


# ------------------------------------------------------------ our arm ----------

def run_ours(args, rank, world):
    import torch

    import w4a8_quantized_gemm_gb300 as eg
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", rank)) if world > 1 else 0)
    torch.cuda.set_device(dev)
    eg.load()
    path = {"auto": eg.PATH_AUTO, "gemv": eg.PATH_GEMV, "tc": eg.PATH_TC}[args.path]
    wl = Workload(args.workload, dev, m=args.m, lin=(args.k, args.n), path=path,
                  variant=args.variant, fused=args.fused, api=args.api)
    peaks = load_peaks()
    copies = wl.n_copies
    step_ops = [wl.step_ops(c) for c in range(copies)]
    launches_per_step = len(step_ops[0])

    def step(c):
        for op in step_ops[c]:
            op[7]()

    stream = torch.cuda.Stream(device=dev)
    # warm-up (also sets kernel attributes outside capture), then capture one
    # graph per layer copy
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            step(i % copies)
    stream.synchronize()
    graphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(c)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % copies].replay()
    stream.synchronize()
    assert eg.device_status() == 0

    # ---- timed region: K graph replays, inputs resident -----------------------
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(args.steps):
                graphs[i % copies].replay()
            e1.record(stream)
        stream.synchronize()
        time.sleep(0.2)
    torch.cuda.synchronize()
    ms_total = e0.elapsed_time(e1)
    if world > 1:
        ms_total = max_over_ranks(ms_total, dev)
    ms_step = ms_total / args.steps
    per_step_bytes = sum(op[5] for op in step_ops[0])
    per_step_ops = sum(op[6] for op in step_ops[0])
    unit_is_ops = ops_unit(args)
    per_step_units = per_step_ops if unit_is_ops else per_step_bytes
    value = per_step_units * args.steps * world / (ms_total * 1e-3) / (1e12 if unit_is_ops else 1e9)

    # ---- per-kernel durations: for each kernel, a CUDA graph of just its
    # launches in the step (per layer copy), replayed over K steps and timed
    # with events on the launching stream -------------------------------------
    per_kernel = {}
    labels = sorted(set(kernel_label(eg, op[1], op[2], path) for op in step_ops[0]))
    for lab in labels:
        sub_graphs, nbytes, nops, nl = [], 0, 0, 0
        for c in range(copies):
            sel = [op for op in step_ops[c] if kernel_label(eg, op[1], op[2], path) == lab]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for op in sel:
                    op[7]()
            sub_graphs.append(g)
            if c == 0:
                nbytes, nops, nl = (sum(op[5] for op in sel), sum(op[6] for op in sel), len(sel))
        with torch.cuda.stream(stream):
            for i in range(3):
                sub_graphs[i % copies].replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(args.steps):
                sub_graphs[i % copies].replay()
            b.record(stream)
        stream.synchronize()
        per_kernel[lab] = {"ms": a.elapsed_time(b), "bytes": nbytes * args.steps,
                           "ops": nops * args.steps, "launches": nl * args.steps}
    dom_name, dom = max(per_kernel.items(), key=lambda kv: kv[1]["ms"])
    if dom_name.startswith("tc_gemm") and unit_is_ops:
        achieved = dom["ops"] / (dom["ms"] * 1e-3) / 1e12
        # fp16 kind::f16 MMA: same nominal rate as bf16
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops_sustained"]}
    else:
        achieved = dom["bytes"] / (dom["ms"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    roof.update({"kernel": dom_name, "traffic": measured_traffic(args, dom_name),
                 "peak_source": peaks["source"],
                 "avg_launch_us": dom["ms"] * 1e3 / dom["launches"]})

    # ---- end to end through the API: each step copies its activations from
    # pinned host memory, replays the captured step (the same API calls) and
    # copies its outputs back to pinned host memory ----------------------------
    ins, outs = wl.host_io()
    h2d = sum(h.numel() * h.element_size() for h, _ in ins)
    d2h = sum(h.numel() * h.element_size() for _, h in outs)
    torch.cuda.synchronize()

    def e2e_step(i):
        for h, d in ins:
            d.copy_(h, non_blocking=True)
        graphs[i % copies].replay()
        for d, h in outs:
            h.copy_(d, non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(2):
            e2e_step(i)
    stream.synchronize()
    t0 = time.perf_counter()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e2.record(stream)
        for i in range(args.steps):
            e2e_step(i)
        e3.record(stream)
    stream.synchronize()
    e2e_ms = e2.elapsed_time(e3)
    wall_ms = (time.perf_counter() - t0) * 1e3
    e2e_value = per_step_units * args.steps * world / (max(e2e_ms, wall_ms) * 1e-3) / \
        (1e12 if unit_is_ops else 1e9)
    status = eg.device_status()

    result = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TOPS" if unit_is_ops else "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_string(args),
        "data": "synthetic (seeded splitmix64/Box-Muller; 7B/DiT shapes, random weights)",
        "config": workload_config(args, wl, per_step_bytes, per_step_ops),
        "tops": round(per_step_ops * args.steps * world / (ms_total * 1e-3) / 1e12, 4),
        "gbps": round(per_step_bytes * args.steps * world / (ms_total * 1e-3) / 1e9, 2),
        "roofline": {k: (round(v, 4) if isinstance(v, float) else v) for k, v in roof.items()},
        "per_kernel": {k: {"launches": v["launches"], "ms": round(v["ms"], 4),
                           "GB/s": round(v["bytes"] / (v["ms"] * 1e-3) / 1e9, 1),
                           "TOPS": round(v["ops"] / (v["ms"] * 1e-3) / 1e12, 2)}
                       for k, v in per_kernel.items()},
        "e2e": {"value": round(e2e_value, 3), "unit": "TOPS" if unit_is_ops else "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(max(e2e_ms, wall_ms) / args.steps, 5)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "path": args.path,
        "device_status": status,
    }
    if args.twin:
        twin = measure_twin(args, wl, step_ops, stream, unit_is_ops)
        if twin is not None:
            twin["int4_kernels_ms_per_step"] = round(
                sum(v["ms"] for k, v in per_kernel.items() if k.startswith(("tc_gemm", "gemv_w4")))
                / args.steps, 5)
            result["bf16_twin"] = twin
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args, wl, unit_is_ops, budget_s=args.cpu_budget)
    return result


def measure_twin(args, wl, step_ops, stream, unit_is_ops):
    """The dense bf16 twin: every int4 product of the step on weights
    dequantized once to bf16 (egopq_dequant_w4), each run as a plain cuBLAS
    bf16 GEMM (torch.matmul) on the same bf16 activations -- the speed a
    dequantize-once path gets, and the dense-GEMM yardstick for the packed
    kernels. Timed like the main leg: one CUDA graph per layer copy, K replays."""
    import torch

    eg = wl.eg
    dense, t_dq = {}, 0.0
    graphs, flops, nbytes = [], 0, 0
    for c in range(wl.n_copies):
        specs = wl.twin_specs.get(c, [])
        for (_, M, N, K, xd, packed, y) in specs:
            key = packed.data_ptr()
            if key not in dense:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    a.record(stream)
                    dense[key] = eg.dequant_w4(packed, N, K, stream=stream)
                    b.record(stream)
                stream.synchronize()
                t_dq += a.elapsed_time(b)
        if c == 0:
            flops = sum(2 * M * N * K for (_, M, N, K, *_r) in specs)
            nbytes = sum(2 * N * K + 2 * M * K + 2 * M * N for (_, M, N, K, *_r) in specs)
    if not flops:
        return None
    outs = {}
    with torch.cuda.stream(stream):
        for c in range(wl.n_copies):
            for (lab, M, N, K, xd, packed, y) in wl.twin_specs[c]:
                torch.matmul(xd, dense[packed.data_ptr()].t(), out=y)  # warm-up, cuBLAS heuristics
    stream.synchronize()
    for c in range(wl.n_copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for (lab, M, N, K, xd, packed, y) in wl.twin_specs[c]:
                torch.matmul(xd, dense[packed.data_ptr()].t(), out=y)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for i in range(3):
            graphs[i % len(graphs)].replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            graphs[i % len(graphs)].replay()
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    dense_bytes = sum(t.numel() * 2 for t in dense.values())
    del dense, outs, graphs
    torch.cuda.empty_cache()
    return {"kernel": "cuBLAS bf16 GEMM (torch.matmul) on weights dequantized once by "
                      "egopq_dequant_w4",
            "value": round((flops if unit_is_ops else nbytes) / (ms * 1e-3)
                           / (1e12 if unit_is_ops else 1e9), 3),
            "unit": "TFLOP/s" if unit_is_ops else "GB/s (bf16 weights)",
            "ms_per_step": round(ms, 5), "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
            "products_per_step": sum(len(v) for v in wl.twin_specs.values()) // max(1, wl.n_copies),
            "dequant_once_ms": round(t_dq, 3), "dense_weight_bytes": dense_bytes}


def dtype_string(args) -> str:
    v = args.variant if args.workload == "linear" else ("w4a16" if args.workload == "dit" else "w4a8")
    return {"w4a8": "int8 x int4 -> exact int32 group partials, f32 combine, bf16 out",
            "w8a8": "int8 x int8 -> exact int32 sums, f32 combine, bf16 out",
            "w4a16": "bf16 x int4/int8 -> f32, bf16 out" if args.workload == "dit"
                     else "bf16 x int4 -> f32, bf16 out",
            "w8a16": "bf16 x int8 -> f32, bf16 out"}[v]


def ops_unit(args) -> bool:
    """Tensor-core-sized workloads (more than 64 tokens) report TOPS, the rest
    GB/s."""
    return args.workload == "prefill" or (args.workload in ("linear", "model") and args.m > 64)


def workload_description(args) -> str:
    return {
        "decode": "decode GEMV sweep: Qwen2.5-7B q,k,v,o,gate,up,down (K=3584/18944), "
                  "M in {1,4,16}, int4 asym group 128, per-token int8 activations",
        "prefill": "prefill W4A8 GEMM: the seven 7B linears + untied head (N=152064), "
                   "M in {512,2048,4096}",
        "model": f"full 7B linear pass: 28 layers x 7 linears + head at M={args.m}",
        "dit": "weight-only W4A16 and W8A16 on DiT blocks K=3072/12288, M in {1,16,4096}",
        "tiny": "tiny W4A8: M=16, K=512, N=256",
        "linear": f"one {args.variant.upper()} linear K={args.k} N={args.n} at M={args.m}"
                  + (" (per-token int8 activations, per-channel int8 weights)"
                     if args.variant == "w8a8" else ""),
    }[args.workload]


def workload_config(args, wl, per_step_bytes, per_step_ops):
    cfg = {"workload": workload_description(args)}
    cfg.update({"layer_copies": wl.n_copies, "bytes_per_step": per_step_bytes,
                "int_ops_per_step": per_step_ops,
                "l2_defeat": "weights rotated across layer copies larger than L2"
                             if wl.n_copies > 1 or args.workload == "model"
                             else "per-step weights larger than L2" if args.workload == "prefill"
                             else "small (L2 resident)",
                "graphs": "one CUDA graph per layer copy",
                "fused_siblings": bool(args.fused), "api": args.api})
    return cfg


# ------------------------------------------------------ oracle (CPU) arm ----------

def cpu_baseline(args, wl, unit_is_ops, budget_s=20.0):
    """Time the CPU oracle as it stands on a bounded sample of the workload."""
    import oracle
    import synth
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    oracle.build()
    done_units, elapsed, samples = 0, 0.0, []
    ops = [op for op in wl.step_ops(0) if op[1] != "quant"]
    # bounded sample: at most 8 rows of each linear and as many columns as
    # make one call last about target_s (the column count adapts to the
    # measured speed of the previous call); passes over the step's linears
    # until the budget is spent
    target_s = max(0.05, budget_s / (2 * max(1, len(ops))))
    ops_per_s = 2e9  # first guess, corrected after every call
    i = 0
    while elapsed < budget_s or not samples:
        op = ops[i % len(ops)]
        i += 1
        label, kind, M, N, K = op[0], op[1], op[2], op[3], op[4]
        m = min(M, 8)
        n = int(target_s * ops_per_s / max(1, 2 * m * K))
        n = min(N, max(128, (n // 128) * 128))
        w = synth.w4_weights(1, 0, 0, n, K)
        x = synth.activations(1, 0, 0, m, K)
        if kind in ("w8a16", "w8a8"):
            w8, s8 = synth.w8_weights(4, 0, 0, n, K)
        t0 = time.perf_counter()
        if kind == "w4a8":
            a_q, a_s, _ = oracle.quant_act(x)
            oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
            nbytes = w4a8_bytes(m, n, K)
        elif kind == "w4a16":
            oracle.w4a16(x, w.w_q, w.scale_f16, w.zero)
            nbytes = w4a16_bytes(m, n, K)
        elif kind == "w8a8":
            a_q, a_s, _ = oracle.quant_act(x)
            oracle.w8a8(a_q, a_s, w8, s8)
            nbytes = w8a8_bytes(m, n, K)
        else:
            oracle.w8a16(x, w8, s8)
            nbytes = w8a16_bytes(m, n, K)
        units = 2 * m * n * K if unit_is_ops else nbytes
        dt = time.perf_counter() - t0
        ops_per_s = 2 * m * n * K / max(dt, 1e-6)
        elapsed += dt
        done_units += units
        samples.append(f"{label}: {m}x{n}x{K}")
    value = done_units / elapsed / (1e12 if unit_is_ops else 1e9)
    return {"value": round(value, 5), "unit": "TOPS" if unit_is_ops else "GB/s", "cores": cores,
            "kind": "oracle", "seconds": round(elapsed, 2),
            "sample": f"{len(samples)} oracle GEMMs on row/column subsets of the step's linears "
                      f"(<=8 tokens, columns sized to at most ~{target_s:.2f} s a call): "
                      + "; ".join(samples[:8])
                      + ("; ..." if len(samples) > 8 else "")}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, timed as it stands, rank 0 only."""
    if rank != 0:
        return None

    class _WL:  # shapes only; no GPU
        pass
    wl = _WL()
    wl.n_copies = 1
    unit_is_ops = ops_unit(args)
    shapes = {"decode": [(M, K, N) for M in (1, 4, 16) for (_, K, N) in SHAPES_7B],
              "prefill": [(M, K, N) for M in (512, 2048, 4096) for (_, K, N) in SHAPES_7B + [HEAD]],
              "model": [(args.m, K, N) for (_, K, N) in SHAPES_7B] + [(args.m, HEAD[1], HEAD[2])],
              "dit": [(M, K, N) for M in (1, 16, 4096) for (K, N) in
                      [(3072, 3072), (3072, 12288), (12288, 3072)]],
              "tiny": [(16, 512, 256)],
              "linear": [(args.m, args.k, args.n)]}[args.workload]
    kind = args.variant if args.workload == "linear" else (
        "w4a16" if args.workload == "dit" else "w4a8")
    wl.step_ops = lambda c: [(f"M={M} K={K} N={N}", kind, M, N, K, 0, 0, None)
                             for (M, K, N) in shapes]
    # each step a bounded sample of the workload, sized so that the whole
    # warm-up + timed run stays within about two minutes
    per_step_s = min(5.0, max(0.05, 120.0 / max(1, args.steps + args.warmup)))
    if args.warmup > 0:
        cpu_baseline(args, wl, unit_is_ops, budget_s=per_step_s * args.warmup)  # warm-up
    t0 = time.perf_counter()
    base = cpu_baseline(args, wl, unit_is_ops, budget_s=per_step_s * args.steps)
    wall = time.perf_counter() - t0
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": base["value"],
        "unit": base["unit"],
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(wall * 1e3 / max(1, args.steps), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int64 / fp64 (oracle)",
        "data": "synthetic (seeded splitmix64/Box-Muller; 7B/DiT shapes, random weights)",
        "config": {"workload": workload_description(args),
                   "arm": "CPU oracle on a bounded sample of each step"},
        "cpu_baseline": base,
        "e2e": {"value": base["value"], "unit": base["unit"], "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about half a second of work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["decode", "prefill", "model", "dit", "tiny", "linear"],
                    default="decode")
    ap.add_argument("--m", type=int, default=1, help="tokens for --workload model / linear")
    ap.add_argument("--k", type=int, default=3584, help="K for --workload linear")
    ap.add_argument("--n", type=int, default=3584, help="N for --workload linear")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--twin", action="store_true",
                    help="also time the dense bf16 twin: the step's int4 products as cuBLAS "
                         "bf16 GEMMs on weights dequantized once")
    ap.add_argument("--path", choices=["auto", "gemv", "tc"], default="auto")
    ap.add_argument("--variant", choices=["w4a8", "w4a16", "w8a16", "w8a8"], default="w4a8",
                    help="variant for --workload linear")
    ap.add_argument("--api", choices=["gemm", "linear"], default="gemm",
                    help="gemm: egopq_quant_act_i8 + egopq_w4a8_gemm per linear input; "
                         "linear: one egopq_w4a8_linear call per linear")
    ap.add_argument("--fused", action="store_true",
                    help="run q|k|v and gate|up as one GEMM each (same weights, same outputs)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = {"decode": 1500, "model": 200, "tiny": 2000, "linear": 200}.get(
            args.workload, 40) if args.impl == "ours" else 3
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
