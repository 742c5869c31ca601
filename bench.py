"""Benchmark of the W4A8 packed-linear path on GB300 (one JSON line on stdout).

Workloads (synthetic, seeded; shapes of Qwen2.5-7B linears and DiT blocks):
  sweep    (default) one step = the decode part then the prefill part below,
           i.e. the seven 7B linears at M in {1, 4, 16} and, with the untied
           output head, at M in {512, 2048, 4096}: the metric's M = 1..4096.
  decode   per-token int8 quantization of each linear input + the seven W4A8
           linears q,k,v,o,gate,up,down at M in {1, 4, 16}; four layer copies
           rotate so the weights streamed per step exceed L2.
  prefill  the same seven linears plus the untied quantized output head
           (K=3584, N=152064) at M in {512, 2048, 4096}.
  model    the full linear pass: 28 layers x 7 = 196 W4A8 linears + head at
           one M (--m), independent weights per layer.
  dit      W4A16 and W8A16 on K=3072,N in {3072,12288} and K=12288,N=3072 at
           M in {1, 16, 4096}.
  tiny     M=16, K=512, N=256 (the oracle-sized case).
  linear   one linear of --k/--n at --m tokens (--variant), for profiling.

Sibling linears that read one input (q|k|v, gate|up) run as ONE grouped
library call by default (--api grouped); --api gemm runs one call per linear,
--api linear the one-call quantize+GEMM per linear, --fused concatenated
weights.

value = algorithmic integer ops per second (TOPS) of the whole step for the
        sweep and the tensor-core-sized workloads, algorithmic bytes per second
        (GB/s) for decode-sized ones; K timed steps, inputs resident in HBM.
e2e   = the same through the public API with each step's activations copied
        from pinned host memory and its outputs copied back (on copy streams of
        their own, overlapping the neighbouring steps' compute).
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
from dataclasses import dataclass
from typing import Callable, Optional

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A8 GEMM TOPS and HBM GB/s (% of roofline) on 7B-shaped linears, M=1–4096"
SHAPES_7B = [("q", 3584, 3584), ("k", 3584, 512), ("v", 3584, 512), ("o", 3584, 3584),
             ("gate", 3584, 18944), ("up", 3584, 18944), ("down", 18944, 3584)]
HEAD = ("head", 3584, 152064)
INPUT_OF = {"q": "attn", "k": "attn", "v": "attn", "o": "o", "gate": "mlp", "up": "mlp",
            "down": "down", "head": "head"}
INPUT_K = {"attn": 3584, "o": 3584, "mlp": 3584, "down": 18944, "head": 3584}
INPUT_SEED = {"attn": 0, "o": 3, "mlp": 4, "down": 6, "head": 7}
SIBLINGS = {"qkv": ["q", "k", "v"], "gate_up": ["gate", "up"]}
G128 = 128
# layer copies per part (rotated step to step so that weights stream from HBM)
COPIES = {"decode": 4, "prefill": 1, "model": 1, "dit": 1, "tiny": 1, "linear": 1}
# seed config index of each part's weights and activations
SEED_CONFIG = {"tiny": 0, "decode": 1, "prefill": 2, "model": 3, "dit": 4, "linear": 1}


# ------------------------------------------------------------ algorithmic work --

def w4a8_bytes(M, N, K):
    G = K // G128
    return N * K // 2 + 2 * N * G + N * G // 2 + M * K + 4 * M + 4 * M * G + 2 * M * N


def w4a8_tc_actual_bytes(M, N, K):
    """What the tensor-core path reads instead: the 2-byte-per-code operand
    form of the activations (two e4m3 planes or fp16 codes) in place of the
    int8 codes."""
    return w4a8_bytes(M, N, K) + M * K


def quant_bytes(M, K):
    return 2 * M * K + M * K + 4 * M + 4 * M * (K // G128)


def quant_actual_bytes(M, K, with_tc=True, with_codes=True):
    """What the quantizer writes in place of the algorithmic int8 codes: the
    int8 codes where a GEMV reads them, the tensor-core operand form (2 bytes
    a code) where the tensor-core path reads it."""
    codes = (M * K if with_codes else 0) + (2 * M * K if with_tc else 0)
    return quant_bytes(M, K) - M * K + codes


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


# ------------------------------------------------------------------ the plan --
# A step is a list of parts; a part a list of cells (one library call each),
# laid out from the shapes alone so that both arms describe the same work.

@dataclass
class Cell:
    label: str              # e.g. "gate M=2048", "quant mlp M=16", "qkv M=1"
    kind: str               # quant | w4a8 | w4a16 | w8a16 | w8a8
    M: int
    N: int                  # output rows (sum over grouped siblings)
    K: int
    inp: str                # activation it reads
    names: tuple            # linears it computes
    bytes: int              # algorithmic bytes
    ops: int                # algorithmic integer ops (flops for weight-only)
    with_quant: bool = False  # one-call linear: its quantization is in this cell
    layer: int = 0          # layer of the model pass


def part_names(args):
    return ["decode", "prefill"] if args.workload == "sweep" else [args.workload]


def plan_part(args, part):
    """Cells of one part, in launch order."""
    cells = []
    api = args.api

    def add_w4a8(M, names, K, N, inp, first_of_input, layer):
        sib = next((k for k, v in SIBLINGS.items() if v == list(names)), None)
        label = f"{sib or names[0]} M={M}" + (f" L{layer}" if part == "model" else "")
        if api == "linear":
            # the one-call linear quantizes its input itself (once per input:
            # the first cell reading it carries the quantization's bytes)
            qb = quant_bytes(M, K) if first_of_input else 0
            cells.append(Cell(label, "w4a8", M, N, K, inp, tuple(names),
                              w4a8_bytes(M, N, K) + qb, 2 * M * N * K, with_quant=True,
                              layer=layer))
            return
        cells.append(Cell(label, "w4a8", M, N, K, inp, tuple(names), w4a8_bytes(M, N, K),
                          2 * M * N * K, layer=layer))

    if part in ("decode", "prefill", "tiny", "linear", "model"):
        if part == "decode":
            ms, shapes = [1, 4, 16], list(SHAPES_7B)
        elif part == "prefill":
            ms, shapes = [512, 2048, 4096], list(SHAPES_7B) + [HEAD]
        elif part == "model":
            ms, shapes = [args.m], list(SHAPES_7B)
        elif part == "linear":
            ms, shapes = [args.m], [("q", args.k, args.n)]
        else:
            ms, shapes = [16], [("q", 512, 256)]
        layers = 28 if part == "model" else 1
        group = (api in ("grouped", "linear") or args.fused) and \
            part in ("decode", "prefill", "model")
        for M in ms:
            for layer in range(layers):
                done = set()
                i = 0
                while i < len(shapes):
                    nm, K, N = shapes[i]
                    inp = INPUT_OF.get(nm, "attn") if part not in ("tiny", "linear") else "attn"
                    sib = next((s for s in SIBLINGS.values() if s[0] == nm), None) if group else None
                    names = sib if sib else [nm]
                    Ntot = sum(n for (x, _, n) in shapes if x in names) if sib else N
                    first = inp not in done
                    if api != "linear" and first:
                        cells.append(Cell(f"quant {inp} M={M}", "quant", M, 0, K, inp, (),
                                          quant_bytes(M, K), 0, layer=layer))
                    done.add(inp)
                    add_w4a8(M, names, K, Ntot, inp, first, layer)
                    i += len(names)
            if part == "model":
                nm, K, N = HEAD
                if api != "linear":
                    cells.append(Cell(f"quant head M={M}", "quant", M, 0, K, "head", (),
                                      quant_bytes(M, K), 0))
                add_w4a8(M, ["head"], K, N, "head", True, 0)
        if part == "linear" and args.variant != "w4a8":
            cells = []
            M, K, N = args.m, args.k, args.n
            if args.variant == "w8a8":
                cells.append(Cell(f"quant M={M}", "quant", M, 0, K, "attn", (), quant_bytes(M, K), 0))
            fn = {"w4a16": w4a16_bytes, "w8a16": w8a16_bytes, "w8a8": w8a8_bytes}[args.variant]
            cells.append(Cell(f"{args.variant} K={K} N={N} M={M}", args.variant, M, N, K, "attn",
                              ("q",), fn(M, N, K), 2 * M * N * K))
    elif part == "dit":
        for M in (1, 16, 4096):
            for (K, N) in [(3072, 3072), (3072, 12288), (12288, 3072)]:
                cells.append(Cell(f"w4a16 K={K} N={N} M={M}", "w4a16", M, N, K, f"dit{K}", ("w4",),
                                  w4a16_bytes(M, N, K), 2 * M * N * K))
                cells.append(Cell(f"w8a16 K={K} N={N} M={M}", "w8a16", M, N, K, f"dit{K}", ("w8",),
                                  w8a16_bytes(M, N, K), 2 * M * N * K))
    else:
        raise ValueError(part)
    return cells


def ops_unit(args) -> bool:
    """TOPS for the sweep and tensor-core-sized workloads (more than 64 tokens),
    GB/s for the rest."""
    return (args.workload in ("sweep", "prefill")
            or (args.workload in ("linear", "model") and args.m > 64))


def workload_description(args) -> str:
    d = {
        "sweep": "7B-shaped W4A8 linears at M=1..4096: decode part (q,k,v,o,gate,up,down at "
                 "M in {1,4,16}) + prefill part (the same seven + untied head N=152064 at "
                 "M in {512,2048,4096}); int4 asym group 128, per-token int8 activations",
        "decode": "decode sweep: Qwen2.5-7B q,k,v,o,gate,up,down (K=3584/18944), "
                  "M in {1,4,16}, int4 asym group 128, per-token int8 activations",
        "prefill": "prefill W4A8 GEMM: the seven 7B linears + untied head (N=152064), "
                   "M in {512,2048,4096}",
        "model": f"full 7B linear pass: 28 layers x 7 linears + head at M={args.m}",
        "dit": "weight-only W4A16 and W8A16 on DiT blocks K=3072/12288, M in {1,16,4096}",
        "tiny": "tiny W4A8: M=16, K=512, N=256",
        "linear": f"one {args.variant.upper()} linear K={args.k} N={args.n} at M={args.m}",
    }
    return d[args.workload]


def workload_config(args) -> dict:
    """The `config` object, from the plan alone (both arms print the same)."""
    parts = part_names(args)
    cfg = {"workload": workload_description(args)}
    per_bytes = per_ops = 0
    for p in parts:
        cells = plan_part(args, p)
        per_bytes += sum(c.bytes for c in cells)
        per_ops += sum(c.ops for c in cells)
    cfg.update({
        "parts": parts,
        "layer_copies": {p: COPIES[p] for p in parts},
        "bytes_per_step": per_bytes, "int_ops_per_step": per_ops,
        "l2_defeat": ("decode weights rotated across 4 layer copies (484 MB); prefill "
                      "weights 404 MB per step" if args.workload == "sweep" else
                      "weights rotated across layer copies larger than L2"
                      if COPIES.get(args.workload, 1) > 1 or args.workload == "model"
                      else "per-step weights larger than L2" if args.workload == "prefill"
                      else "small (L2 resident)"),
        "graphs": "one CUDA graph per part and layer copy",
        "api": args.api, "fused_siblings": bool(args.fused), "path": args.path,
    })
    return cfg


def dtype_string(args) -> str:
    v = args.variant if args.workload == "linear" else ("w4a16" if args.workload == "dit" else "w4a8")
    return {"w4a8": "int8 x int4 -> exact int32 group partials, f32 combine, bf16 out",
            "w8a8": "int8 x int8 -> exact int32 sums, f32 combine, bf16 out",
            "w4a16": "bf16 x int4/int8 -> f32, bf16 out" if args.workload == "dit"
                     else "bf16 x int4 -> f32, bf16 out",
            "w8a16": "bf16 x int8 -> f32, bf16 out"}[v]


# --------------------------------------------------------- DRAM traffic table --

def _code_only(text: str) -> str:
    """The source with its comments and blank lines taken out (trailing
    whitespace too): what a change to the counters can come from."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_sources_hash() -> str:
    """sha256 over the CUDA sources and the public header (names and code,
    comments left out: a comment edit does not invalidate measured traffic)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "w4a8_quantized_gemm_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc)
                   if f.endswith((".cu", ".cuh", ".h")))
    files.append(os.path.join(ROOT, "include", "egopq.h"))
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()


def traffic_table():
    """{(kernel label, M, N, K): DRAM bytes of one call (all its launches of
    that kernel)} from the ncu
    captures summarised in profiles/dram_traffic.txt, or {} when there is none
    or the kernels changed since they were taken (source hash mismatch)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return {}
    table, want = {}, None
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line.startswith("sources_sha256="):
                want = line.split("=", 1)[1]
            elif line.startswith("kernel="):
                fields = dict(kv.split("=", 1) for kv in line.split("\t"))
                table[(fields["kernel"], int(fields["M"]), int(fields["N"]), int(fields["K"]))] = \
                    float(fields["bytes"])
    if want is None or want != kernel_sources_hash():
        return {}
    return table


def measured_traffic(table, label, cells, launches):
    """Average DRAM bytes per launch of kernel `label` over the step's cells
    (launches[i]: launches of cells[i]), or None unless every cell's shape was
    captured."""
    total = 0.0
    for c in cells:
        key = (label, c.M, c.N, c.K)
        if key not in table:
            return None
        total += table[key]
    return total / sum(launches) if cells else None


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


# ---------------------------------------------------------------- GPU side ----

def _to_dev(torch, a, dev, dt=None):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a).to(dev)
    return t.view(dt) if dt is not None else t


def kernel_label(eg, cell: Cell, path: int) -> str:
    kind, M = cell.kind, cell.M
    if kind == "quant":
        return "quant_act_kernel"
    variant = {"w4a8": eg.VARIANT_W4A8, "w4a16": eg.VARIANT_W4A16, "w8a16": eg.VARIANT_W8A16,
               "w8a8": eg.VARIANT_W8A8}[kind]
    use = path if path != eg.PATH_AUTO else eg.auto_path(M, variant)
    if use == eg.PATH_GEMV:
        return {"w4a8": "gemv_w4_kernel (W4A8)", "w4a16": "gemv_w4_kernel (W4A16)",
                "w8a16": "gemv_w8_kernel (W8A16)", "w8a8": "gemv_w8a8_kernel (W8A8)"}[kind]
    if kind == "w4a8":
        return ("tc_gemm_kernel (W4A8, e4m3 tiles)"
                if eg.tc_operand_form(M) == eg.TC_FORM_E4M3_PLANES
                else "tc_gemm_kernel (W4A8, fp16 tiles)")
    return f"tc_gemm_kernel ({kind.upper()})"


def kernel_launches(eg, cell: Cell, path: int) -> int:
    """Launches of the cell's kernel (the library's own count on the
    tensor-core path: a long-K persistent grid whose last round would be
    short runs that round as a second, split-K launch)."""
    if cell.kind == "quant" or "tc_gemm" not in kernel_label(eg, cell, path):
        return 1
    variant = {"w4a8": eg.VARIANT_W4A8, "w4a16": eg.VARIANT_W4A16, "w8a16": eg.VARIANT_W8A16,
               "w8a8": eg.VARIANT_W8A8}[cell.kind]
    return eg.tc_launches(cell.M, cell.N, cell.K, variant)


def call_launches(eg, cell: Cell, path: int) -> int:
    """All launches of the cell's library call (the one-call linear also
    launches its quantization)."""
    return kernel_launches(eg, cell, path) + (1 if cell.with_quant else 0)


def actual_bytes(eg, cell: Cell, path: int, tc_inputs=()) -> int:
    """Bytes the launch moves: the algorithmic bytes, plus the tensor-core
    operand form of the activations where that path writes or reads it."""
    if cell.kind == "quant":
        key = (cell.M, cell.inp)
        return quant_actual_bytes(cell.M, cell.K, key in tc_inputs, key not in tc_inputs)
    if cell.kind == "w4a8" and "tc_gemm" in kernel_label(eg, cell, path):
        # the one-call linear on this path writes the 2-byte operand form and
        # no int8 codes: one byte a code more than the algorithmic count
        extra = cell.M * cell.K \
            if cell.with_quant and cell.bytes > w4a8_bytes(cell.M, cell.N, cell.K) else 0
        return cell.bytes + cell.M * cell.K + extra
    return cell.bytes


class Part:
    """One part of the step on the GPU: weights for each layer copy, inputs,
    outputs and one callable per cell, bound to the plan."""

    def __init__(self, args, name, dev, path):
        import torch

        import synth
        import w4a8_quantized_gemm_gb300 as eg
        self.torch, self.eg, self.dev, self.name, self.path = torch, eg, dev, name, path
        self.cells = plan_part(args, name)
        self.copies = COPIES[name]
        cfg = SEED_CONFIG[name]
        t = lambda a, dt=None: _to_dev(torch, a, dev, dt)
        self.layer_count = 28 if name == "model" else 1
        self.args = args
        # weights: packs[copy][(layer, linear)] (one packed tensor per linear;
        # --fused concatenates siblings into one)
        self.packs = []
        self.w8 = {}
        if name == "dit":
            for (K, N) in [(3072, 3072), (3072, 12288), (12288, 3072)]:
                w = synth.w4_weights(cfg, 0, 0, N, K)
                w8, s8 = synth.w8_weights(cfg, 0, 0, N, K)
                self.w8[(K, N)] = (eg.pack_w4(t(w.w_q), t(w.scale_f16, torch.float16),
                                              t(w.zero)), t(w8), t(s8, torch.float16))
            self.packs = [None]
        elif name == "linear" and args.variant in ("w8a16", "w8a8", "w4a16"):
            K, N = args.k, args.n
            w = synth.w4_weights(cfg, 0, 0, N, K)
            w8, s8 = synth.w8_weights(cfg, 0, 0, N, K)
            self.w8[(K, N)] = (eg.pack_w4(t(w.w_q), t(w.scale_f16, torch.float16), t(w.zero)),
                               t(w8), t(s8, torch.float16))
            self.packs = [None]
        else:
            shapes = {c_nm: None for c in self.cells for c_nm in c.names}
            all_shapes = dict((nm, (K, N)) for (nm, K, N) in SHAPES_7B + [HEAD])
            if name in ("tiny", "linear"):
                all_shapes = {"q": (self.cells[-1].K, self.cells[-1].N)}
            for c in range(self.copies):
                packs = {}
                for layer in range(self.layer_count):
                    for nm in shapes:
                        K, N = all_shapes[nm]
                        w = synth.w4_weights(cfg, c * self.layer_count + layer,
                                             synth.LINEARS[nm], N, K)
                        packs[(layer, nm)] = eg.pack_w4(t(w.w_q), t(w.scale_f16, torch.float16),
                                                        t(w.zero))
                if args.fused:
                    for layer in range(self.layer_count):
                        for sib in SIBLINGS.values():
                            if all((layer, s) in packs for s in sib):
                                packs[(layer, "+".join(sib))] = torch.cat(
                                    [packs[(layer, s)] for s in sib])
                self.packs.append(packs)
        torch.cuda.synchronize()
        # activations: one bf16 input per (M, input), one quantized set each:
        # the tensor-core operand form where tensor-core cells read the input,
        # the int8 codes otherwise (a path reads one or the other)
        self.x, self.q = {}, {}
        tc_inputs = {(c.M, c.inp) for c in self.cells
                     if c.kind in ("w4a8", "w8a8") and "tc_gemm" in kernel_label(eg, c, path)}
        gemv_inputs = {(c.M, c.inp) for c in self.cells
                       if c.kind in ("w4a8", "w8a8") and "tc_gemm" not in kernel_label(eg, c, path)}
        assert not (tc_inputs & gemv_inputs), "an input read by both paths"
        for c in self.cells:
            key = (c.M, c.inp)
            if key in self.x:
                continue
            if name == "dit" or (name == "linear" and args.variant != "w4a8"):
                x = synth.activations(cfg, 0, 0, c.M, c.K, outliers=False)
            else:
                x = synth.activations(cfg, 0, INPUT_SEED.get(c.inp, 0), c.M, c.K)
            self.x[key] = t(x, torch.bfloat16)
            self.q[key] = eg.QuantAct(
                torch.empty((c.M, c.K), dtype=torch.int8, device=dev)
                if key not in tc_inputs else None,
                torch.empty((c.M,), dtype=torch.float32, device=dev),
                torch.empty((c.M, c.K // G128), dtype=torch.int32, device=dev),
                eg.tc_operand(c.M, c.K, dev) if key in tc_inputs else None)
        # outputs: one per (cell, linear)
        self.y = {}
        for i, c in enumerate(self.cells):
            if c.kind == "quant":
                continue
            if len(c.names) > 1 and not args.fused:
                Ns = [dict((nm, n) for (nm, _, n) in SHAPES_7B)[nm] for nm in c.names]
                self.y[i] = [torch.empty((c.M, n), dtype=torch.bfloat16, device=dev) for n in Ns]
            else:
                self.y[i] = [torch.empty((c.M, c.N), dtype=torch.bfloat16, device=dev)]
        self.tc_inputs = tc_inputs
        self._ws = {}
        self._pack_io()
        self.fns = [self._bind(copy) for copy in range(self.copies)]

    def _pack_io(self):
        """Every bf16 input in one device buffer and every output in another
        (views keep their shapes; sizes are multiples of 256 bytes, so each view
        stays 16-byte aligned), so that the end-to-end leg moves a step's inputs
        and outputs with one copy each way."""
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

        keys = list(self.x.keys())
        self.x_all, xs = pack([self.x[k] for k in keys])
        self.x = dict(zip(keys, xs))
        flat = [(i, j) for i in sorted(self.y) for j in range(len(self.y[i]))]
        self.y_all, ys = pack([self.y[i][j] for (i, j) in flat])
        for (i, j), v in zip(flat, ys):
            self.y[i][j] = v

    def second_io_set(self):
        """A second packed input buffer and output buffer with the same layout,
        and the cell callables (per layer copy) bound to them: the end-to-end
        leg copies one step's inputs and outputs while the next step computes
        on the other set. Returns (x_all, y_all, fns)."""
        torch = self.torch

        def views(buf, base_buf, base_views):
            flat = buf.view(-1)
            out = []
            for v in base_views:
                off = (v.data_ptr() - base_buf.data_ptr()) // v.element_size()
                out.append(flat[off:off + v.numel()].view(v.shape))
            return out

        x_all = torch.empty_like(self.x_all)
        x_all.copy_(self.x_all)
        y_all = torch.empty_like(self.y_all)
        keys = list(self.x.keys())
        saved_x, saved_y = self.x, self.y
        self.x = dict(zip(keys, views(x_all, self.x_all, [saved_x[k] for k in keys])))
        self.y = {i: views(y_all, self.y_all, ys) for i, ys in saved_y.items()}
        try:
            fns = [self._bind(copy) for copy in range(self.copies)]
        finally:
            self.x, self.y = saved_x, saved_y
        return x_all, y_all, fns

    def workspace(self, M, K):
        need = self.eg.w4a8_linear_workspace_bytes(M, K, self.path)
        if (M, K) not in self._ws:
            self._ws[(M, K)] = self.torch.empty(need, dtype=self.torch.uint8, device=self.dev)
        return self._ws[(M, K)]

    def _bind(self, copy):
        """One callable per cell for layer copy `copy`."""
        eg, args, path = self.eg, self.args, self.path
        fns = []
        for i, c in enumerate(self.cells):
            key = (c.M, c.inp)
            xd, a = self.x[key], self.q[key]
            if c.kind == "quant":
                fns.append(lambda xd=xd, a=a: eg.quant_act(xd, out=a))
                continue
            ys = self.y[i]
            if self.name in ("dit",) or c.kind in ("w4a16", "w8a16", "w8a8"):
                p4, w8, s8 = self.w8[(c.K, c.N)]
                f = {"w4a16": lambda xd=xd, p=p4, c=c, y=ys[0]: eg.w4a16_gemm(
                         xd, p, c.N, c.K, out=y, path=path),
                     "w8a16": lambda xd=xd, w8=w8, s8=s8, y=ys[0]: eg.w8a16_gemm(
                         xd, w8, s8, out=y, path=path),
                     "w8a8": lambda a=a, w8=w8, s8=s8, y=ys[0]: eg.w8a8_gemm(
                         a, w8, s8, out=y, path=path)}[c.kind]
                fns.append(f)
                continue
            layer = c.layer
            packs = self.packs[copy]
            if len(c.names) > 1 and args.fused:
                p = packs[(layer, "+".join(c.names))]
                fns.append(lambda a=a, p=p, c=c, y=ys[0]: eg.w4a8_gemm(a, p, c.N, c.K, out=y,
                                                                      path=path))
            elif len(c.names) > 1:
                ps = [packs[(layer, nm)] for nm in c.names]
                Ns = [y.shape[1] for y in ys]
                if args.api == "linear":
                    ws = self.workspace(c.M, c.K)
                    fns.append(lambda xd=xd, ps=ps, Ns=Ns, ys=ys, ws=ws: eg.w4a8_linear_grouped(
                        xd, ps, Ns, path=path, out=ys, workspace=ws))
                else:
                    fns.append(lambda a=a, ps=ps, Ns=Ns, c=c, ys=ys: eg.w4a8_gemm_grouped(
                        a, ps, Ns, c.K, path=path, out=ys))
            else:
                p = packs[(layer, c.names[0])]
                if args.api == "linear":
                    ws = self.workspace(c.M, c.K)
                    fns.append(lambda xd=xd, p=p, c=c, y=ys[0], ws=ws: eg.w4a8_linear(
                        xd, p, c.N, out=y, workspace=ws, path=path))
                else:
                    fns.append(lambda a=a, p=p, c=c, y=ys[0]: eg.w4a8_gemm(a, p, c.N, c.K, out=y,
                                                                          path=path))
        return fns

    def run(self, copy, select=None):
        for i, f in enumerate(self.fns[copy]):
            if select is None or i in select:
                f()


def measure_int8_yardstick(torch, dev):
    """Dense int8 tensor-core GEMM through the library (cuBLASLt, via
    torch._int_mm: int8 x int8 -> int32) on a 7B-shaped product, best of three
    timed runs of 10 calls."""
    M, N, K = 4096, 18944, 3584
    try:
        A = torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev)
        B = torch.randint(-127, 128, (N, K), dtype=torch.int8, device=dev)
        for _ in range(3):
            torch._int_mm(A, B.t())
        torch.cuda.synchronize()
        best = 1e30
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(10):
                torch._int_mm(A, B.t())
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b) / 10)
        del A, B
        return {"tops": round(2 * M * N * K / (best * 1e-3) / 1e12, 1),
                "shape": f"{M}x{N}x{K}",
                "how": "cuBLASLt int8 GEMM (torch._int_mm, int32 out), best of 3 x 10 calls"}
    except Exception as e:  # a library without an int8 kernel for this device
        return {"tops": None, "how": f"torch._int_mm unavailable: {str(e)[:120]}"}


def measure_twin(parts, stream, steps, torch, eg):
    """Dense comparisons on the step's tensor-core-sized W4A8 products (more
    than 64 tokens), each weight dequantized once to bf16 by egopq_dequant_w4:
    the same products as cuBLAS bf16 GEMMs (torch.matmul), as the structure
    twin (egopq_bf16_gemm_twin: the W4A16 pipeline with a copy in place of the
    int4 unpack), and as the W4A16 kernel on the packed weights -- all on the
    same bf16 activations. Each leg is one CUDA graph, K replays."""
    prods = []
    for p in parts:
        for i, c in enumerate(p.cells):
            if c.kind != "w4a8" or c.M <= 64:
                continue
            Ns = [y.shape[1] for y in p.y[i]] if len(p.y[i]) > 1 else [c.N]
            for nm, n in zip(c.names if len(Ns) > 1 else c.names[:1], Ns):
                key = (c.layer, nm) if not (p.args.fused and len(c.names) > 1) else None
                packed = p.packs[0][key] if key else p.packs[0][(c.layer, "+".join(c.names))]
                prods.append((c.M, n, c.K, p.x[(c.M, c.inp)], packed))
    if not prods:
        return None
    dense, t_dq = {}, 0.0
    for (M, N, K, xd, packed) in prods:
        if packed.data_ptr() not in dense:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                dense[packed.data_ptr()] = eg.dequant_w4(packed, N, K, stream=stream)
                b.record(stream)
            stream.synchronize()
            t_dq += a.elapsed_time(b)
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device=xd.device)
            for (M, N, K, xd, _) in prods]
    legs = {
        "cublas_bf16": lambda: [torch.matmul(xd, dense[pk.data_ptr()].t(), out=o)
                                for (M, N, K, xd, pk), o in zip(prods, outs)],
        "structure_twin_bf16": lambda: [eg.bf16_gemm_twin(xd, dense[pk.data_ptr()], out=o)
                                        for (M, N, K, xd, pk), o in zip(prods, outs)],
        "w4a16_packed": lambda: [eg.w4a16_gemm(xd, pk, N, K, out=o, path=eg.PATH_TC)
                                 for (M, N, K, xd, pk), o in zip(prods, outs)],
    }
    flops = sum(2 * M * N * K for (M, N, K, _, _) in prods)
    res = {}
    for name, fn in legs.items():
        with torch.cuda.stream(stream):
            fn()  # warm-up (library heuristics, kernel attributes)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(steps):
                g.replay()
            b.record(stream)
        stream.synchronize()
        ms = a.elapsed_time(b) / steps
        res[name] = {"ms_per_step": round(ms, 4), "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1)}
        del g
    res["products"] = len(prods)
    res["dequant_once_ms"] = round(t_dq, 3)
    res["how"] = ("the step's W4A8 products above 64 tokens on bf16 activations: cuBLAS and the "
                  "structure twin on weights dequantized once, W4A16 on the packed weights")
    del dense, outs
    torch.cuda.empty_cache()
    return res


def _roofline(label, ms, nbytes, nops, launches, peaks, int8, traffic):
    # the bound that binds: tensor where the kernel's work has more ops per
    # byte than the ridge of the two measured peaks, HBM otherwise
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    tensor = nops / max(nbytes, 1) > ridge
    if tensor:
        achieved = nops / (ms * 1e-3) / 1e12
        r = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops_sustained"],
             "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops_sustained"],
             "peak_kind": "dense bf16 cuBLAS, sustained (kind::f16 MMA, same nominal rate)"}
        if int8 and int8.get("tops"):
            r["frac_of_int8_peak"] = achieved / int8["tops"]
    else:
        achieved = nbytes / (ms * 1e-3) / 1e9
        r = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
             "frac": achieved / peaks["hbm_gbs"], "peak_kind": "HBM copy"}
    r.update({"kernel": label, "traffic": traffic, "algorithmic_bytes_per_launch":
              nbytes / launches, "peak_source": peaks["source"],
              "avg_launch_us": ms * 1e3 / launches})
    return {k: (round(v, 4) if isinstance(v, float) else v) for k, v in r.items()}


def run_ours(args, rank, world):
    import torch

    import w4a8_quantized_gemm_gb300 as eg
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", rank)) if world > 1 else 0)
    torch.cuda.set_device(dev)
    eg.load()
    path = {"auto": eg.PATH_AUTO, "gemv": eg.PATH_GEMV, "tc": eg.PATH_TC}[args.path]
    peaks = load_peaks()
    parts = [Part(args, nm, dev, path) for nm in part_names(args)]
    unit_is_ops = ops_unit(args)
    stream = torch.cuda.Stream(device=dev)

    # warm-up (also sets kernel attributes outside capture), then one graph per
    # part and layer copy
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            for p in parts:
                p.run(i % p.copies)
    stream.synchronize()
    for p in parts:
        p.graphs = []
        for c in range(p.copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                p.run(c)
            p.graphs.append(g)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            for p in parts:
                p.graphs[i % p.copies].replay()
    stream.synchronize()
    assert eg.device_status() == 0

    # ---- timed region: K steps of graph replays, inputs resident; an event
    # after each part splits the time by part -------------------------------
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    marks = [[torch.cuda.Event(enable_timing=True) for _ in parts] for _ in range(args.steps)]
    with ClockSampler(dev.index) as clk:
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for i in range(args.steps):
                for pi, p in enumerate(parts):
                    p.graphs[i % p.copies].replay()
                    marks[i][pi].record(stream)
        stream.synchronize()
        time.sleep(0.2)
    torch.cuda.synchronize()
    ms_total = ev0.elapsed_time(marks[-1][-1])
    part_ms = [0.0] * len(parts)
    prev = ev0
    for i in range(args.steps):
        for pi in range(len(parts)):
            part_ms[pi] += prev.elapsed_time(marks[i][pi])
            prev = marks[i][pi]
    if world > 1:
        ms_total = max_over_ranks(ms_total, dev)
    ms_step = ms_total / args.steps
    per_step_bytes = sum(c.bytes for p in parts for c in p.cells)
    per_step_ops = sum(c.ops for p in parts for c in p.cells)
    per_step_units = per_step_ops if unit_is_ops else per_step_bytes
    scale = 1e12 if unit_is_ops else 1e9
    value = per_step_units * args.steps * world / (ms_total * 1e-3) / scale

    # ---- per kernel: for each part and kernel, a CUDA graph of just that
    # kernel's launches in the step (per layer copy), replayed over K steps and
    # timed with events on the launching stream ------------------------------
    per_kernel, kernel_cells = {}, {}
    for p in parts:
        labels = sorted(set(kernel_label(eg, c, path) for c in p.cells))
        for lab in labels:
            sel = {i for i, c in enumerate(p.cells) if kernel_label(eg, c, path) == lab}
            sub = []
            for c in range(p.copies):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    p.run(c, sel)
                sub.append(g)
            with torch.cuda.stream(stream):
                for i in range(3):
                    sub[i % p.copies].replay()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for i in range(args.steps):
                    sub[i % p.copies].replay()
                b.record(stream)
            stream.synchronize()
            cs = [p.cells[i] for i in sorted(sel)]
            d = per_kernel.setdefault(lab, {"ms": 0.0, "bytes": 0, "actual": 0, "ops": 0,
                                            "launches": 0})
            d["ms"] += a.elapsed_time(b)
            d["bytes"] += sum(c.bytes for c in cs) * args.steps
            d["actual"] += sum(actual_bytes(eg, c, path, p.tc_inputs) for c in cs) * args.steps
            d["ops"] += sum(c.ops for c in cs) * args.steps
            d["launches"] += sum(kernel_launches(eg, c, path) for c in cs) * args.steps
            kernel_cells.setdefault(lab, []).extend(cs)
            del sub

    # ---- per cell: each library call alone, K replays ------------------------
    cells_out = {}
    if args.cells:
        for p in parts:
            for i, cell in enumerate(p.cells):
                if cell.kind == "quant":
                    continue
                sub = []
                for c in range(p.copies):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        p.run(c, {i})
                    sub.append(g)
                reps = max(args.steps, 20)
                with torch.cuda.stream(stream):
                    for r in range(3):
                        sub[r % p.copies].replay()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    for r in range(reps):
                        sub[r % p.copies].replay()
                    b.record(stream)
                stream.synchronize()
                us = a.elapsed_time(b) * 1e3 / reps
                gbs = cell.bytes / (us * 1e-6) / 1e9
                tops = cell.ops / (us * 1e-6) / 1e12
                fh = gbs / peaks["hbm_gbs"]
                ft = tops / peaks["bf16_tflops_sustained"]
                cells_out[f"{p.name}: {cell.label}"] = {
                    "us": round(us, 2), "GB/s": round(gbs, 1), "TOPS": round(tops, 2),
                    "frac_hbm": round(fh, 3), "frac_tensor": round(ft, 3),
                    "bound": "hbm" if fh >= ft else "tensor",
                    "kernel": kernel_label(eg, cell, path)}
                del sub

    int8 = measure_int8_yardstick(torch, dev) if unit_is_ops else None
    table = traffic_table()

    def roof(lab):
        d = per_kernel[lab]
        return _roofline(lab, d["ms"], d["bytes"], d["ops"], d["launches"], peaks, int8,
                         measured_traffic(table, lab, kernel_cells[lab],
                                          [kernel_launches(eg, c, path)
                                           for c in kernel_cells[lab]]))

    gemm_labels = [k for k in per_kernel if not k.startswith("quant")]
    dom = max(per_kernel, key=lambda k: per_kernel[k]["ms"])
    roofline = roof(dom)
    hbm_labels = [k for k in gemm_labels if roof(k)["bound"] == "hbm"]

    # ---- end to end through the API: each step copies its activations from
    # pinned host memory, replays the captured step (the same API calls) and
    # copies its outputs back to pinned host memory. The copies run on their
    # own streams, so that step i's outputs travel back (and step i+1's inputs
    # in) while the next step computes: each part has two device input/output
    # sets used by alternate steps, and events order every copy against the
    # compute that produces or reads its set. Every step's copies are inside
    # the timed region. ----------------------------------------------------------
    for p in parts:
        x_b, y_b, fns_b = p.second_io_set()
        p.io_sets = [(p.x_all, p.y_all, p.graphs)]
        saved = p.fns
        p.fns = fns_b
        graphs_b = []
        for c in range(p.copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                p.run(c)
            graphs_b.append(g)
        p.fns = saved
        p.io_sets.append((x_b, y_b, graphs_b))
        p.xh = torch.empty(p.x_all.shape, dtype=p.x_all.dtype).pin_memory()
        p.xh.copy_(p.x_all.cpu())
        p.yh = torch.empty(p.y_all.shape, dtype=p.y_all.dtype).pin_memory()
    h2d = sum(p.xh.numel() * p.xh.element_size() for p in parts)
    d2h = sum(p.yh.numel() * p.yh.element_size() for p in parts)
    torch.cuda.synchronize()
    h2d_s = torch.cuda.Stream(device=dev)
    d2h_s = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of set b landed
    ev_comp = [torch.cuda.Event() for _ in range(2)]   # compute on set b done
    ev_out = [torch.cuda.Event() for _ in range(2)]    # outputs of set b read back

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(h2d_s):
            if i >= 2:
                h2d_s.wait_event(ev_comp[b])   # step i-2 has read these inputs
            for p in parts:
                p.io_sets[b][0].copy_(p.xh, non_blocking=True)
            ev_in[b].record(h2d_s)
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])   # step i-2's outputs are back
            for p in parts:
                p.io_sets[b][2][i % p.copies].replay()
            ev_comp[b].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev_comp[b])
            for p in parts:
                p.yh.copy_(p.io_sets[b][1], non_blocking=True)
            ev_out[b].record(d2h_s)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    h2d_s.wait_event(e2)
    d2h_s.wait_event(e2)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_event(ev_out[(args.steps - 1) % 2])
    if args.steps > 1:
        stream.wait_event(ev_out[args.steps % 2])
    e3.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e2.elapsed_time(e3)
    wall_ms = (time.perf_counter() - t0) * 1e3
    e2e_value = per_step_units * args.steps * world / (max(e2e_ms, wall_ms) * 1e-3) / scale
    status = eg.device_status()

    parts_out = {}
    for p, ms in zip(parts, part_ms):
        pb = sum(c.bytes for c in p.cells)
        po = sum(c.ops for c in p.cells)
        sec = ms * 1e-3 / args.steps
        d = {"ms_per_step": round(ms / args.steps, 5), "GB/s": round(pb / sec / 1e9, 1),
             "TOPS": round(po / sec / 1e12, 2), "frac_hbm": round(pb / sec / 1e9 / peaks["hbm_gbs"], 4),
             "frac_bf16_sustained": round(po / sec / 1e12 / peaks["bf16_tflops_sustained"], 4),
             "launches_per_step": sum(call_launches(eg, c, path) for c in p.cells)}
        if int8 and int8.get("tops"):
            d["x_int8_peak"] = round(po / sec / 1e12 / int8["tops"], 3)
        parts_out[p.name] = d

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
        "config": workload_config(args),
        "tops": round(per_step_ops * args.steps * world / (ms_total * 1e-3) / 1e12, 4),
        "gbps": round(per_step_bytes * args.steps * world / (ms_total * 1e-3) / 1e9, 2),
        "parts": parts_out,
        "roofline": roofline,
        "roofline_decode": roof(max(hbm_labels, key=lambda k: per_kernel[k]["ms"]))
        if hbm_labels and len(parts) > 1 else None,
        "rooflines": {k: {kk: vv for kk, vv in roof(k).items()
                          if kk in ("bound", "achieved", "unit", "frac", "traffic",
                                    "avg_launch_us")} for k in gemm_labels},
        "int8_yardstick": int8,
        "per_kernel": {k: {"launches": v["launches"], "ms": round(v["ms"], 4),
                           "GB/s": round(v["bytes"] / (v["ms"] * 1e-3) / 1e9, 1),
                           "actual_GB/s": round(v["actual"] / (v["ms"] * 1e-3) / 1e9, 1),
                           "TOPS": round(v["ops"] / (v["ms"] * 1e-3) / 1e12, 2),
                           "share_of_kernel_time": round(v["ms"] / sum(
                               x["ms"] for x in per_kernel.values()), 4)}
                       for k, v in per_kernel.items()},
        "cells": cells_out or None,
        "e2e": {"value": round(e2e_value, 3), "unit": "TOPS" if unit_is_ops else "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(max(e2e_ms, wall_ms) / args.steps, 5),
                "how": "pinned host buffers; each step's inputs in and outputs out on "
                       "copy streams of their own, overlapping the neighbouring steps' "
                       "compute (two device input/output sets, used by alternate steps)"},
        "gpu_launches": sum(call_launches(eg, c, path) for p in parts for c in p.cells)
        * args.steps,
        "clocks": clk.summary(),
        "device_status": status,
    }
    if args.twin:
        result["twin"] = measure_twin(parts, stream, args.steps, torch, eg)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args, unit_is_ops, budget_s=args.cpu_budget)
    return result


# ------------------------------------------------------ oracle (CPU) arm ----------

def cpu_baseline(args, unit_is_ops, budget_s=20.0):
    """Time the CPU oracle as it stands on a bounded sample of the workload:
    at most 8 rows of each GEMM cell of the plan and as many columns as make
    one call last about target_s (adapted to the measured speed), cycling over
    the cells until the budget is spent."""
    import oracle
    import synth
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    oracle.build()
    cells = [c for p in part_names(args) for c in plan_part(args, p) if c.kind != "quant"]
    done_units, elapsed, samples = 0, 0.0, []
    target_s = max(0.05, budget_s / (2 * max(1, len(cells))))
    ops_per_s = 2e9  # first guess, corrected after every call
    i = 0
    while elapsed < budget_s or not samples:
        c = cells[i % len(cells)]
        i += 1
        m, K = min(c.M, 8), c.K
        n = int(target_s * ops_per_s / max(1, 2 * m * K))
        n = min(c.N, max(128, (n // 128) * 128))
        w = synth.w4_weights(1, 0, 0, n, K)
        x = synth.activations(1, 0, 0, m, K)
        if c.kind in ("w8a16", "w8a8"):
            w8, s8 = synth.w8_weights(4, 0, 0, n, K)
        t0 = time.perf_counter()
        if c.kind == "w4a8":
            a_q, a_s, _ = oracle.quant_act(x)
            oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
            nbytes = w4a8_bytes(m, n, K)
        elif c.kind == "w4a16":
            oracle.w4a16(x, w.w_q, w.scale_f16, w.zero)
            nbytes = w4a16_bytes(m, n, K)
        elif c.kind == "w8a8":
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
        samples.append(f"{c.label}: {m}x{n}x{K}")
    value = done_units / elapsed / (1e12 if unit_is_ops else 1e9)
    return {"value": round(value, 5), "unit": "TOPS" if unit_is_ops else "GB/s", "cores": cores,
            "kind": "oracle", "seconds": round(elapsed, 2),
            "sample": f"{len(samples)} oracle GEMMs on row/column subsets of the step's cells "
                      f"(<=8 tokens, columns sized to at most ~{target_s:.2f} s a call): "
                      + "; ".join(samples[:8])
                      + ("; ..." if len(samples) > 8 else "")}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, timed as it stands, rank 0 only."""
    if rank != 0:
        return None
    unit_is_ops = ops_unit(args)
    # each step a bounded sample of the workload, sized so that the whole
    # warm-up + timed run stays within about two minutes
    per_step_s = min(5.0, max(0.05, 120.0 / max(1, args.steps + args.warmup)))
    if args.warmup > 0:
        cpu_baseline(args, unit_is_ops, budget_s=per_step_s * args.warmup)  # warm-up
    t0 = time.perf_counter()
    base = cpu_baseline(args, unit_is_ops, budget_s=per_step_s * args.steps)
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
        "config": workload_config(args),
        "arm": "CPU oracle on a bounded sample of each step",
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
    ap.add_argument("--workload", choices=["sweep", "decode", "prefill", "model", "dit", "tiny",
                                           "linear"], default="sweep")
    ap.add_argument("--m", type=int, default=1, help="tokens for --workload model / linear")
    ap.add_argument("--k", type=int, default=3584, help="K for --workload linear")
    ap.add_argument("--n", type=int, default=3584, help="N for --workload linear")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cells", dest="cells", action="store_false",
                    help="skip timing each library call of the step alone")
    ap.add_argument("--twin", action="store_true",
                    help="also time the dense comparisons (cuBLAS bf16, the structure twin, "
                         "W4A16) on the step's tensor-core-sized products")
    ap.add_argument("--path", choices=["auto", "gemv", "tc"], default="auto")
    ap.add_argument("--variant", choices=["w4a8", "w4a16", "w8a16", "w8a8"], default="w4a8",
                    help="variant for --workload linear")
    ap.add_argument("--api", choices=["grouped", "gemm", "linear"], default="grouped",
                    help="grouped: one quantization per input + one grouped GEMM per set of "
                         "sibling linears; gemm: one GEMM call per linear; linear: the one-call "
                         "quantize+GEMM (grouped for siblings)")
    ap.add_argument("--fused", action="store_true",
                    help="run q|k|v and gate|up as one GEMM each on concatenated weights")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = {"sweep": 30, "decode": 1500, "model": 200, "tiny": 2000,
                      "linear": 200}.get(args.workload, 40) if args.impl == "ours" else 3
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
