"""Benchmark of the BitDelta hot path on GB300.

Default workload (one GPU): the 70B-FFN-shaped decode GEMV -- W_base bf16
[28672 x 8192] ~ N(0, 0.02), Delta ~ Laplace(0, 1e-3), per-row alpha -- where
one step is the whole path over one batch: bd_compress (Delta, sign bits,
alpha) followed by the fused linear for 1, 4 and 16 tokens.  The metric is
HBM GB/s of algorithmic bytes per step; the JSON line also carries tokens/s,
the roofline of the dominant kernel (CUDA-event timed inside the timed
region), the CPU oracle timed on the host cores, an end-to-end number with
host buffers, and the SM clocks sampled during the timed region.

Other workloads (--workload): tiny (256x256, T=4, per-matrix alpha), multi
(8192x8192 shared W_base, 14 variants, 64 Zipf-routed tokens) and prefill
(4096 tokens x 8192x8192, the tensor-core path, reported in TFLOP/s).  The
default decode line also carries a short prefill measurement under
"prefill", since the metric names prefill TFLOP/s.  slice: the 8-layer slice of
a 70B-shaped stack (56 linears, 14 variants compressed on the GPU, 32 decode
tokens routed by Zipf), one step = the 56 multi-variant linears.

`python bench.py --impl reference` times the CPU oracle instead (the
reference arm), on bounded samples of the same workload.

Multi-GPU: one process per GPU (torchrun); every rank runs its own copy of
the workload (the path has no exchange step), the timed region is bracketed
by barriers and the slowest rank's time is reported (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import threading
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused BitDelta linear HBM GB/s (% of peak), tokens/s; prefill TFLOP/s (% peak)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch from
# one ncu capture, keyed by kernel; each entry records the sha256 of the
# kernel's source file at capture time and is ignored once that source has
# changed.  Summaries of the captures are in profiles/.  An entry whose value
# is a float is a ratio (traffic / algorithmic bytes) taken on one launch of a
# smaller call of the same kernel and applied to the average launch.
NCU_TRAFFIC = {
    # (kernel, workload): (source sha256[:16], source file, bytes per launch or ratio)
    ("skinny_kernel<1>", "decode"): ("60707ad3c65224a0", "bd_skinny.cu", 499_405_056 + 3_889_920),
    # 4 rows per CTA (kCompressRowsPerCta in bd_internal.h)
    ("compress_kernel", "decode"): ("364b9a156a18e55b", "bd_compress.cu", 939_566_080 + 7_655_936),
    ("prefill_kernel", "prefill"): ("705a6fbf4f52e879", "bd_prefill.cu", 591_238_912 + 67_592_704),
    # multi_kernel only (the prepare pass adds about 3.7 MB of x tiles and corrections)
    ("multi_prepare + multi_kernel<8>", "multi"): ("d89f83fcd4e67914", "bd_multi.cu", 255_770_880 + 3_986_432),
    # the grouped prefill_kernel only (router, plan and gather add about 134 MB of x copies)
    ("route + gather + prefill_kernel (grouped)", "multi_prefill"): ("705a6fbf4f52e879", "bd_prefill.cu",
                                                                      1_097_012_736 + 64_569_088),
    ("materialize_kernel", "materialize"): ("fae23fcd0ba90d9b", "bd_materialize.cu", 499_370_496 + 426_232_320),
}


# kernels each timed call launches: multi = prepare + fused kernel; multi_prefill =
# router + plan + gather + grouped prefill; slice = 56 multi calls
LAUNCHES_PER_CALL = {"multi": 2, "slice": 2, "multi_prefill": 4, "monosoup": 88}
# workloads whose own figure is tensor throughput (TFLOP/s) rather than GB/s
TENSOR_WORKLOADS = ("prefill", "multi_prefill")
# workloads bound by fp32 CUDA-core arithmetic: their figure is fp32 TFLOP/s
ALU_WORKLOADS = ("monosoup",)
# fp32 FMA peak of the GB300 from unit counts: 152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
# MonoSoup workload: k checkpoints, rank r, sketch width l, power iterations q
MONOSOUP = {"d": 8192, "k": 3, "rank": 16, "l": 32, "q": 1}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--workload", choices=["decode", "tiny", "multi", "prefill", "multi_prefill", "materialize", "monosoup",
                                          "slice"], default="decode")
    p.add_argument("--no-prefill", action="store_true", help="skip the prefill sub-measurement of the decode line")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    return p.parse_args()


def _src_sha(name: str) -> str:
    path = os.path.join(ROOT, "bit_weight_delta_bd_gb300", "csrc", name)
    with open(path, "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            pk = json.load(fh)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ----------------------------------------------------------------------------- workloads

def materialize_bytes(d_out, d_in, n_alpha):
    """W_base read, W_eff written (2 bytes each per weight), bits and alpha read."""
    return 4 * d_out * d_in + d_out * d_in // 8 + 4 * n_alpha


def monosoup_bytes(d, k, q):
    """Each pass over a task vector reads W_i and W_base (2 + 2q + ... passes:
    sketch, 2q power-iteration products, B^T), plus the merge's W_base read
    and W_merged write."""
    return k * (2 + 2 * q) * 4 * d * d + 4 * d * d


def monosoup_flops(d, k, rank, l, q):
    """fp32 FLOPs of the products with the task vectors (2 d^2 l each) and of
    the rank-(k r) merge (2 d^2 k r)."""
    return k * (2 + 2 * q) * 2 * d * d * l + 2 * d * d * k * rank


def linear_bytes(T, d_out, d_in, n_alpha, y_bytes=2):
    """Algorithmic bytes of one fused linear: W_base + bits + alpha + x + y."""
    return 2 * d_out * d_in + d_out * d_in // 8 + 4 * n_alpha + 2 * T * d_in + y_bytes * T * d_out


def compress_bytes(d_out, d_in, n_alpha):
    """Algorithmic bytes of one compression: W_base + W_ft read, bits + alpha written."""
    return 4 * d_out * d_in + d_out * d_in // 8 + 4 * n_alpha


class Workload:
    """Host inputs (numpy bf16 bits) plus the list of calls of one step."""

    def __init__(self, name, seed):
        from bit_weight_delta_bd_gb300 import synth

        self.name = name
        if name == "slice":  # weights are drawn on the device by SliceRun
            self.tokens = [32]
            self.per_row = True
            self.vid = synth.zipf_variant_ids(np.random.default_rng(seed), 32, 14)
            self.d_out = self.d_in = 0
            self.wf, self.xs, self.wb = [None] * 14, [], None
            self.n_alpha = 0
            return
        if name in ("decode", "tiny"):
            d_out, d_in = (28672, 8192) if name == "decode" else (256, 256)
            self.tokens = [1, 4, 16] if name == "decode" else [4]
            self.per_row = name == "decode"
            rng = np.random.default_rng(seed)
            self.wb = synth.base_weight(rng, d_out, d_in)
            self.wf = [synth.finetuned_weight(rng, self.wb, 1e-3)]
            self.xs = [synth.activations(rng, T, d_in) for T in self.tokens]
            self.vid = None
        elif name == "materialize":
            d_out, d_in = 28672, 8192
            self.tokens = []
            self.per_row = True
            self.wb, wf, _ = synth.single_problem(seed, d_out, d_in, 1)
            self.wf = [wf]
            self.xs = []
            self.vid = None
        elif name == "monosoup":
            d_out = d_in = MONOSOUP["d"]
            self.tokens = []
            self.per_row = True
            self.wb, self.wf = synth.monosoup_checkpoints(seed, d_out, d_in, MONOSOUP["k"], MONOSOUP["rank"])
            self.omega = synth.gaussian_test_matrix(seed + 1, d_in, MONOSOUP["l"])
            self.xs = []
            self.vid = None
        elif name == "prefill":
            d_out, d_in = 8192, 8192
            self.tokens = [4096]
            self.per_row = True
            self.wb, wf, x = synth.single_problem(seed + 3, d_out, d_in, 4096)
            self.wf = [wf]
            self.xs = [x]
            self.vid = None
        else:  # multi (64 tokens, decode kernel) or multi_prefill (4096 tokens, tensor cores)
            d_out, d_in = 8192, 8192
            self.tokens = [4096 if name == "multi_prefill" else 64]
            self.per_row = True
            self.wb, self.wf, x, self.vid, _ = synth.multi_problem(seed, d_out, d_in, self.tokens[0], 14)
            self.xs = [x]
        self.d_out, self.d_in = d_out, d_in
        self.n_alpha = d_out if self.per_row else 1

    def config(self):
        c = {"workload": self.name, "d_out": self.d_out, "d_in": self.d_in, "tokens": self.tokens,
             "alpha": "per_row" if self.per_row else "per_matrix"}
        if self.name == "decode":
            c["workload"] = "decode_ffn_28672x8192_T1_4_16"
            c["step"] = "bd_compress + bd_linear at T=1, 4, 16 (one variant)"
            c["l2"] = "inputs larger than L2 (W_base 470 MB, W_ft 470 MB vs 126.5 MB L2)"
        elif self.name == "slice":
            c = {"workload": "slice_8_layers_70b_shapes_V14_T32", "layers": 8,
                 "linears": "q/o 8192x8192, k/v 8192->1024, gate/up 8192->28672, down 28672->8192",
                 "variants": 14, "active_variants": int(len(set(int(v) for v in self.vid))), "tokens": [32],
                 "alpha": "per_row",
                 "step": "56 bd_linear_multi calls (variants compressed on the GPU once, untimed)",
                 "l2": "inputs larger than L2 (13.7 GB of W_base per step)"}
        elif self.name == "prefill":
            c["workload"] = "prefill_4096x8192x8192"
            c["step"] = "bd_linear at T=4096, one variant (compressed once, untimed); tensor-core path"
            c["l2"] = "inputs larger than L2 (W_base 134 MB + x 67 MB + y 67 MB vs 126.5 MB L2)"
        elif self.name == "multi_prefill":
            c["workload"] = "multi_prefill_8192x8192_V14_T4096"
            c["variants"] = len(self.wf)
            c["active_variants"] = int(len(set(int(v) for v in self.vid)))
            c["step"] = ("bd_linear_multi over 4096 Zipf(1.1)-routed tokens: router, gather, grouped tensor-core "
                         "prefill (variants compressed once, untimed)")
            c["l2"] = "inputs larger than L2 (W_base 134 MB + x 67 MB + y 67 MB vs 126.5 MB L2)"
        elif self.name == "materialize":
            c["workload"] = "materialize_ffn_28672x8192"
            c["step"] = "bd_materialize: W_eff = RN_bf16(W_base + alpha s) written to HBM (variant compressed once, untimed)"
            c["l2"] = "inputs larger than L2 (W_base 470 MB in, W_eff 470 MB out vs 126.5 MB L2)"
        elif self.name == "monosoup":
            c = {"workload": f"monosoup_{self.d_out}x{self.d_in}_k{MONOSOUP['k']}_r{MONOSOUP['rank']}",
                 "d_out": self.d_out, "d_in": self.d_in, **{k: v for k, v in MONOSOUP.items() if k != "d"},
                 "step": ("bd_monosoup_merge: randomized rank-16 truncated SVD of 3 task vectors (sketch width 32, "
                          "one power iteration) and the merge W_base + mean tau_i, bf16 out"),
                 "l2": "inputs larger than L2 (4 x 134 MB of bf16 weights)"}
        elif self.name == "tiny":
            c["workload"] = "tiny_256x256_T4"
            c["step"] = "bd_compress + bd_linear at T=4"
            c["l2"] = "L2-resident (139 KB): latency only, no roofline claim"
        else:
            c["workload"] = "multi_tenant_8192x8192_V14_T64"
            c["variants"] = len(self.wf)
            c["active_variants"] = int(len(set(int(v) for v in self.vid)))
            c["step"] = "bd_linear_multi over 64 Zipf(1.1)-routed tokens (variants compressed once, untimed)"
            c["l2"] = "L2 flushed (256 MB write) before each step; flush excluded from kernel events"
        return c


class GpuRun:
    """Device copies of a workload and the calls of one step."""

    def __init__(self, wl: Workload, dev):
        import torch

        from bit_weight_delta_bd_gb300 import bitdelta as bd

        self.bd, self.torch, self.wl, self.dev = bd, torch, wl, dev
        PR = bd.BD_ALPHA_PER_ROW if wl.per_row else bd.BD_ALPHA_PER_MATRIX
        self.mode = PR

        def d(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

        self.wb = d(wl.wb)
        self.wf = [d(w) for w in wl.wf]
        self.xs = [d(x) for x in wl.xs]
        self.signs = [torch.empty((wl.d_out, wl.d_in // 32), dtype=torch.int32, device=dev) for _ in wl.wf]
        self.alpha = [torch.empty(wl.n_alpha, dtype=torch.float32, device=dev) for _ in wl.wf]
        self.ys = [torch.empty((T, wl.d_out), dtype=torch.bfloat16, device=dev) for T in wl.tokens]
        self.ws = bd.new_workspace(max(bd.bd_compress_workspace_size(wl.d_out, wl.d_in, PR),
                                       bd.bd_linear_workspace_size(64, wl.d_out, wl.d_in),
                                       bd.bd_linear_multi_workspace_size(max(64, max(wl.tokens, default=0)), max(len(wl.wf), 1),
                                                                         wl.d_out, wl.d_in)), dev)
        self.vid = None if wl.vid is None else torch.from_numpy(wl.vid).to(dev)
        self.flush = None
        if wl.name == "materialize":
            self.w_eff = torch.empty((wl.d_out, wl.d_in), dtype=torch.int16, device=dev)
        if wl.name == "monosoup":
            self.omega = torch.from_numpy(wl.omega).to(dev)
            self.w_merged = torch.empty((wl.d_out, wl.d_in), dtype=torch.bfloat16, device=dev)
            self.ws_ms = bd.new_workspace(bd.bd_monosoup_workspace_size(wl.d_out, wl.d_in, len(wl.wf),
                                                                        MONOSOUP["rank"], MONOSOUP["l"]), dev)
        if wl.name in ("multi", "prefill", "multi_prefill", "materialize"):
            for v in range(len(wl.wf)):  # variants are compressed once, before timing
                bd.bd_compress(self.wb, self.wf[v], PR, self.signs[v], self.alpha[v], self.ws)
            torch.cuda.synchronize()
            self.wf = []  # W_ft is not needed any more
            torch.cuda.empty_cache()
        if wl.name == "multi":
            self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def calls(self):
        """[(label, kernel name, algorithmic bytes, flops, fn)] of one step."""
        bd, wl = self.bd, self.wl
        out = []
        if wl.name in ("multi", "multi_prefill"):
            active = sorted(set(int(v) for v in wl.vid if v >= 0))
            T = wl.tokens[0]
            nbytes = (2 * wl.d_out * wl.d_in + len(active) * (wl.d_out * wl.d_in // 8 + 4 * wl.n_alpha) +
                      2 * T * wl.d_in + 2 * T * wl.d_out + 4 * T)
            kname = ("route + gather + prefill_kernel (grouped)" if wl.name == "multi_prefill"
                     else "multi_prepare + multi_kernel<8>")
            flops = 2 * T * wl.d_out * wl.d_in if wl.name == "multi_prefill" else 4 * T * wl.d_out * wl.d_in
            out.append((f"linear_multi_T{T}", kname, nbytes, flops,
                        lambda: bd.bd_linear_multi(self.xs[0], self.vid, self.signs, self.alpha, self.mode, self.wb,
                                                   self.ys[0], self.ws)))
            return out
        if wl.name == "monosoup":
            m = MONOSOUP
            out.append(("monosoup_merge", "bd_monosoup_merge (sketch, transpose-product, Gram, merge kernels)",
                        monosoup_bytes(wl.d_out, len(wl.wf), m["q"]),
                        monosoup_flops(wl.d_out, len(wl.wf), m["rank"], m["l"], m["q"]),
                        lambda: bd.bd_monosoup_merge(self.wb, self.wf, m["rank"], m["l"], m["q"], self.omega,
                                                     self.w_merged, self.ws_ms)))
            return out
        if wl.name == "materialize":
            out.append(("materialize", "materialize_kernel", materialize_bytes(wl.d_out, wl.d_in, wl.n_alpha), 0,
                        lambda: bd.bd_materialize(self.wb, self.signs[0], self.alpha[0], self.mode, self.w_eff)))
            return out
        if wl.name == "prefill":
            T = wl.tokens[0]
            out.append((f"linear_T{T}", "prefill_kernel", linear_bytes(T, wl.d_out, wl.d_in, wl.n_alpha),
                        2 * T * wl.d_out * wl.d_in,
                        lambda: bd.bd_linear(self.xs[0], self.wb, self.signs[0], self.alpha[0], self.mode, self.ys[0],
                                             self.ws)))
            return out
        out.append(("compress", "compress_kernel", compress_bytes(wl.d_out, wl.d_in, wl.n_alpha), 0,
                    lambda: bd.bd_compress(self.wb, self.wf[0], self.mode, self.signs[0], self.alpha[0], self.ws)))
        for i, T in enumerate(wl.tokens):
            nt = 1 if T <= 8 else 2 if T <= 16 else 4 if T <= 32 else 8
            out.append((f"linear_T{T}", f"skinny_kernel<{nt}>", linear_bytes(T, wl.d_out, wl.d_in, wl.n_alpha),
                        4 * T * wl.d_out * wl.d_in,
                        (lambda i=i: bd.bd_linear(self.xs[i], self.wb, self.signs[0], self.alpha[0], self.mode,
                                                  self.ys[i], self.ws))))
        return out


class SliceRun:
    """The 8-layer slice resident on the device: per linear W_base and the 14
    variants' packed signs and alpha (compressed here, on the GPU, from
    on-device seeded draws), plus that linear's 32-token input."""

    def __init__(self, wl: Workload, dev, seed: int, layers: int = 8):
        import torch

        from bit_weight_delta_bd_gb300 import bitdelta as bd
        from bit_weight_delta_bd_gb300 import synth

        self.bd, self.torch, self.wl = bd, torch, wl
        V, T = 14, 32
        scales = synth.slice_variant_scales(seed, V)
        ws_bytes = max(max(bd.bd_compress_workspace_size(d_out, d_in, bd.BD_ALPHA_PER_ROW),
                           bd.bd_linear_multi_workspace_size(T, V, d_out, d_in))
                       for _, d_out, d_in in synth.SLICE_LINEARS)
        self.ws = bd.new_workspace(ws_bytes, dev)
        self.vid = torch.from_numpy(wl.vid).to(dev)
        rng = np.random.default_rng(seed + 17)
        self.mats = []
        for layer in range(layers):
            for m, (name, d_out, d_in) in enumerate(synth.SLICE_LINEARS):
                wb = synth.device_base_weight(synth.slice_seed(seed, layer, m), d_out, d_in, dev)
                signs, alphas = [], []
                for v in range(V):
                    wf = synth.device_finetuned_weight(synth.slice_seed(seed, layer, m, v), wb, float(scales[v]))
                    sg = torch.empty((d_out, d_in // 32), dtype=torch.int32, device=dev)
                    al = torch.empty(d_out, dtype=torch.float32, device=dev)
                    bd.bd_compress(wb, wf, bd.BD_ALPHA_PER_ROW, sg, al, self.ws)
                    del wf
                    signs.append(sg)
                    alphas.append(al)
                x = torch.from_numpy(synth.activations(rng, T, d_in).view(np.int16)).to(dev)
                y = torch.empty((T, d_out), dtype=torch.bfloat16, device=dev)
                self.mats.append((f"L{layer}.{name}", d_out, d_in, wb, signs, alphas, x, y))
        torch.cuda.synchronize()
        if bd.bd_check_async(self.ws) != bd.BD_OK:
            raise RuntimeError("asynchronous error while compressing the slice")
        self.flush = None
        self.xs = [mt[6] for mt in self.mats]
        self.ys = [mt[7] for mt in self.mats]

    def calls(self):
        bd, wl = self.bd, self.wl
        active = len(set(int(v) for v in wl.vid if v >= 0))
        T = 32
        out = []
        for label, d_out, d_in, wb, signs, alphas, x, y in self.mats:
            nbytes = 2 * d_out * d_in + active * (d_out * d_in // 8 + 4 * d_out) + 2 * T * d_in + 2 * T * d_out + 4 * T
            out.append((label, "multi_prepare + multi_kernel<4>", nbytes, 4 * T * d_out * d_in,
                        (lambda wb=wb, signs=signs, alphas=alphas, x=x, y=y:
                         bd.bd_linear_multi(x, self.vid, signs, alphas, bd.BD_ALPHA_PER_ROW, wb, y, self.ws))))
        return out


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc, self.lines = None, []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", gpu_id], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()
        t0 = time.time()  # a first sample before the timed region starts
        while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)

    def stop(self):
        if self.proc is None:
            return None
        n0, t0 = len(self.lines), time.time()  # and one after it ends (short regions lie between two samples)
        while len(self.lines) <= n0 and time.time() - t0 < 1.0 and self.proc.poll() is None:
            time.sleep(0.01)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        out = "".join(self.lines)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _smi_id(local: int) -> str:
    """nvidia-smi id of CUDA device `local` (its UUID, so that a remapped
    CUDA_VISIBLE_DEVICES still names the right GPU)."""
    import torch

    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except (AttributeError, RuntimeError):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v for v in vis.split(",") if v.strip()]
        return ids[local] if local < len(ids) else str(local)


# ----------------------------------------------------------------------------- CPU oracle

def oracle_time(wl: Workload, budget_s: float = 12.0, threads: int = 0):
    """Times the CPU oracle (as it stands) on a bounded sample of one step:
    whole steps for a small matrix, growing row blocks of one step for a large
    one, until `budget_s` of wall time is spent.  Returns (GB/s of algorithmic
    bytes, threads used, sample description)."""
    import oracle

    cores = oracle.set_threads(threads)
    d_out, d_in = wl.d_out, wl.d_in
    step_bytes = sum(c[2] for c in _step_bytes_rows(wl))
    if wl.name == "monosoup":
        # the oracle's full SVD on the leading n x n block of each checkpoint,
        # n doubled while the budget allows, scaled to the full size by the
        # SVD's n^3 cost
        n, t_used, t_last = 256, 0.0, 0.0
        while n <= min(d_out, d_in):
            t0 = time.perf_counter()
            oracle.monosoup_merge(wl.wb[:n, :n], [w[:n, :n] for w in wl.wf], MONOSOUP["rank"])
            t_last = time.perf_counter() - t0
            t_used += t_last
            if t_used > budget_s / 4 or 2 * n > min(d_out, d_in):
                break
            n *= 2
        t_full = t_last * (d_out / n) * (d_in / n) * (min(d_out, d_in) / n)
        return (step_bytes / t_full / 1e9, cores,
                f"oracle merge of {len(wl.wf)} checkpoints on the leading {n}x{n} block ({t_last:.2f} s, numpy "
                f"SVD threads), scaled by n^3 to {d_out}x{d_in} ({t_full:.1f} s)")
    if d_out * d_in <= (1 << 20):  # small: whole steps
        n, t_used = 0, 0.0
        while t_used < budget_s or n == 0:
            t0 = time.perf_counter()
            s, a = oracle.compress(wl.wb, wl.wf[0], wl.per_row)
            for x in wl.xs:
                oracle.linear(x, wl.wb, s, a, wl.per_row)
            t_used += time.perf_counter() - t0
            n += 1
        return step_bytes * n / t_used / 1e9, cores, f"{n} whole steps ({t_used:.2f} s on {cores} threads)"
    rows_done, t_used, chunk = 0, 0.0, 16
    while (t_used < budget_s or rows_done == 0) and rows_done < d_out:
        r = np.arange(rows_done, min(d_out, rows_done + chunk), dtype=np.int64)
        t0 = time.perf_counter()
        sfs, afs = [], []
        for wf in wl.wf:
            s, a = oracle.compress_rows(wl.wb, wf, r)
            sf = np.zeros((d_out, d_in // 32), np.uint32)
            af = np.zeros(d_out, np.float32)
            sf[r], af[r] = s, a
            sfs.append(sf)
            afs.append(af)
        if wl.name == "materialize":
            oracle.materialize(wl.wb[r], sfs[0][r], afs[0][r], True)
        elif wl.vid is None:
            for x in wl.xs:
                oracle.linear(x, wl.wb, sfs[0], afs[0], True, rows=r)
        else:
            oracle.linear_multi(wl.xs[0], wl.vid, sfs, afs, True, wl.wb, rows=r)
        t_used += time.perf_counter() - t0
        rows_done += len(r)
        chunk = min(chunk * 2, 4096)
    gbs = step_bytes * rows_done / d_out / t_used / 1e9
    sample = f"{rows_done} of {d_out} rows of one step ({t_used:.2f} s on {cores} threads)"
    return gbs, cores, sample


def _step_bytes_rows(wl: Workload):
    """(label, kernel, bytes) of one step, computable without a GPU."""
    out = []
    if wl.vid is not None:
        active = sorted(set(int(v) for v in wl.vid if v >= 0))
        T = wl.tokens[0]
        out.append(("linear_multi", "", 2 * wl.d_out * wl.d_in + len(active) * (wl.d_out * wl.d_in // 8 + 4 * wl.n_alpha)
                    + 2 * T * wl.d_in + 2 * T * wl.d_out + 4 * T))
        return out
    if wl.name == "materialize":
        return [("materialize", "", materialize_bytes(wl.d_out, wl.d_in, wl.n_alpha))]
    if wl.name == "monosoup":
        return [("monosoup", "", monosoup_bytes(wl.d_out, len(wl.wf), MONOSOUP["q"]))]
    if wl.name != "prefill":
        out.append(("compress", "", compress_bytes(wl.d_out, wl.d_in, wl.n_alpha)))
    for T in wl.tokens:
        out.append((f"linear_T{T}", "", linear_bytes(T, wl.d_out, wl.d_in, wl.n_alpha)))
    return out


# ----------------------------------------------------------------------------- arms

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _step_flops(wl: Workload) -> int:
    """Useful FLOPs of one step of a tensor- or ALU-bound workload: 2 T d_out
    d_in per linear call; the MonoSoup merge's fp32 products."""
    if wl.name == "monosoup":
        return monosoup_flops(wl.d_out, len(wl.wf), MONOSOUP["rank"], MONOSOUP["l"], MONOSOUP["q"])
    return sum(2 * T * wl.d_out * wl.d_in for T in wl.tokens)


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    wl = Workload(args.workload, args.seed)
    step_bytes = sum(c[2] for c in _step_bytes_rows(wl))
    # each step is a bounded sample so that the whole run stays near 90 s of oracle time
    budget = max(0.01, min(12.0, 90.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        oracle_time(wl, budget_s=budget / 4)
    vals = []
    cores, sample = 0, ""
    for _ in range(args.steps):
        gbs, cores, sample = oracle_time(wl, budget_s=budget)
        vals.append(gbs)
    value = statistics.median(vals)
    ms_per_step = step_bytes / (value * 1e9) * 1e3
    unit = "GB/s"
    if wl.name in TENSOR_WORKLOADS or wl.name in ALU_WORKLOADS:  # the same unit as the GPU arm's line
        value = _step_flops(wl) / (ms_per_step * 1e-3) / 1e12
        unit = "TFLOP/s"
    line = {"metric": METRIC, "value": value, "unit": unit, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy; shapes and distributions of the BitDelta serving setup)",
            "config": wl.config(),
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_setup()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__

    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    __graft_entry__.build()  # no-op once built; loads the library on every rank
    from bit_weight_delta_bd_gb300 import bitdelta as bd

    wl = Workload(args.workload, args.seed + rank)
    run = SliceRun(wl, dev, args.seed + rank) if wl.name == "slice" else GpuRun(wl, dev)
    calls = run.calls()
    stream = torch.cuda.current_stream()

    def one_step(evs=None):
        if run.flush is not None:
            run.flush.fill_(1)
        for i, (_, _, _, _, fn) in enumerate(calls):
            if evs is not None:
                evs[i][0].record(stream)
            fn()
            if evs is not None:
                evs[i][1].record(stream)

    for _ in range(max(args.warmup, 3)):
        one_step()
    if bd.bd_check_async(run.ws) != bd.BD_OK:
        raise RuntimeError("asynchronous error during warm-up")
    torch.cuda.synchronize()

    events = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in calls]
              for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(_smi_id(local))
    t_start.record(stream)
    for k in range(args.steps):
        one_step(events[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    if run.flush is not None:  # the L2 flush is not part of the path: count kernel time only
        elapsed_ms = sum(events[k][i][0].elapsed_time(events[k][i][1]) for k in range(args.steps)
                         for i in range(len(calls)))
    if bd.bd_check_async(run.ws) != bd.BD_OK:
        raise RuntimeError("asynchronous error during the timed region")
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())

    step_bytes = sum(c[2] for c in calls)
    ms_per_step = elapsed_ms / args.steps
    value = world * step_bytes / (ms_per_step * 1e-3) / 1e9
    tokens = sum(wl.tokens)
    hbm_peak, bf16_peak, peak_src = load_peaks()

    # per-kernel averages from the events
    per_kernel = {}
    for i, (label, kname, nbytes, flops, _) in enumerate(calls):
        ms = [events[k][i][0].elapsed_time(events[k][i][1]) for k in range(args.steps)]
        e = per_kernel.setdefault(kname, {"launches": 0, "total_ms": 0.0, "bytes": 0, "labels": []})
        e["launches"] += len(ms)
        e["total_ms"] += sum(ms)
        e["bytes"] += nbytes * len(ms)
        e["labels"].append(label)
    dom = max(per_kernel, key=lambda k: per_kernel[k]["total_ms"])
    d = per_kernel[dom]
    avg_ms = d["total_ms"] / d["launches"]
    bytes_per_launch = d["bytes"] / d["launches"]
    achieved = bytes_per_launch / (avg_ms * 1e-3) / 1e9
    traffic = None
    tr = NCU_TRAFFIC.get((dom, wl.name))
    if tr is not None and tr[0] == _src_sha(tr[1]):
        traffic = tr[2] * bytes_per_launch if isinstance(tr[2], float) else tr[2]
    if wl.name in TENSOR_WORKLOADS:
        flops_per_launch = calls[0][3]
        tf = flops_per_launch / (avg_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": dom, "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s",
                    "frac": tf / bf16_peak, "traffic": traffic, "peak_source": f"{peak_src} (bf16_tflops, burst)",
                    "flops_per_launch": flops_per_launch, "avg_launch_us": avg_ms * 1e3}
    elif wl.name in ALU_WORKLOADS:
        flops_per_launch = calls[0][3]
        tf = flops_per_launch / (avg_ms * 1e-3) / 1e12
        roofline = {"bound": "alu", "kernel": dom, "achieved": tf, "peak": FP32_PEAK_TFLOPS, "unit": "TFLOP/s",
                    "frac": tf / FP32_PEAK_TFLOPS, "traffic": traffic,
                    "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz (fp32 FMA)",
                    "flops_per_launch": flops_per_launch, "avg_launch_us": avg_ms * 1e3,
                    "hbm_achieved_gbs": achieved, "hbm_frac": achieved / hbm_peak}
    else:
        roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "traffic": traffic, "peak_source": f"{peak_src} (hbm_gbs)",
                    "bytes_per_launch": bytes_per_launch, "avg_launch_us": avg_ms * 1e3}
    kernels = {k: {"launches": v["launches"], "avg_us": v["total_ms"] / v["launches"] * 1e3,
                   "share": v["total_ms"] / sum(x["total_ms"] for x in per_kernel.values()),
                   "GBps": v["bytes"] / (v["total_ms"] * 1e-3) / 1e9,
                   "frac_hbm": v["bytes"] / (v["total_ms"] * 1e-3) / 1e9 / hbm_peak, "calls": v["labels"]}
               for k, v in per_kernel.items()}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(run, calls, wl, max(3, min(args.steps, 20)), stream)
        if world > 1:
            t = torch.tensor([e2e["ms_per_step"]], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e["ms_per_step"] = float(t.item())
        e2e["value"] = world * step_bytes / (e2e["ms_per_step"] * 1e-3) / 1e9
        if wl.name in TENSOR_WORKLOADS or wl.name in ALU_WORKLOADS:
            e2e["value"] = world * calls[0][3] / (e2e["ms_per_step"] * 1e-3) / 1e12
            e2e["unit"] = "TFLOP/s"

    prefill = None
    if wl.name == "decode" and not args.no_prefill:
        prefill = measure_prefill(dev, args.seed + rank, bf16_peak, peak_src)
        if world > 1:
            t = torch.tensor([prefill["avg_us"]], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            prefill["avg_us"] = float(t.item())
            prefill["tflops"] = world * prefill["flops_per_launch"] / (prefill["avg_us"] * 1e-6) / 1e12
            prefill["frac"] = prefill["tflops"] / world / bf16_peak

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu and wl.name != "slice":
        gbs, cores, sample = oracle_time(wl)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
        if wl.name in TENSOR_WORKLOADS or wl.name in ALU_WORKLOADS:  # in the line's own unit
            cpu["value"] = _step_flops(wl) / (step_bytes / (gbs * 1e9)) / 1e12
            cpu["unit"] = "TFLOP/s"

    if rank == 0:
        unit = "GB/s"
        if wl.name in TENSOR_WORKLOADS or wl.name in ALU_WORKLOADS:  # this workload's own figure is FLOP/s
            value = world * calls[0][3] / (ms_per_step * 1e-3) / 1e12
            unit = "TFLOP/s"
        line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32" if wl.name in ALU_WORKLOADS else "bf16", "accumulate": "f32",
                "data": "synthetic (seeded numpy; shapes and distributions of the BitDelta serving setup)",
                "config": {**wl.config(), "parallelism": f"replicas x{world} (no exchange step)"},
                "tokens_per_s": world * tokens / (ms_per_step * 1e-3),
                "frac_hbm_step": value / world / hbm_peak,
                "roofline": roofline, "kernels": kernels, "prefill": prefill, "cpu_baseline": cpu, "e2e": e2e,
                "clocks": clk, "gpu_launches": LAUNCHES_PER_CALL.get(wl.name, 1) * len(calls) * args.steps}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def measure_prefill(dev, seed, bf16_peak, peak_src, reps=20):
    """Tensor-core prefill on its own: 4096 tokens x W_base [8192 x 8192], one
    variant; median of `reps` CUDA-event-timed calls."""
    import torch

    wl = Workload("prefill", seed)
    run = GpuRun(wl, dev)
    fn = run.calls()[0][4]
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    stream = torch.cuda.current_stream()
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    if run.bd.bd_check_async(run.ws) != run.bd.BD_OK:
        raise RuntimeError("asynchronous error in the prefill measurement")
    us = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3
    flops = 2 * 4096 * 8192 * 8192
    tf = flops / (us * 1e-6) / 1e12
    return {"workload": "prefill_4096x8192x8192", "kernel": "prefill_kernel", "bound": "tensor", "avg_us": us,
            "flops_per_launch": flops, "tflops": tf, "peak": bf16_peak, "frac": tf / bf16_peak,
            "peak_source": f"{peak_src} (bf16_tflops, burst)", "reps": reps}


def run_e2e(run: GpuRun, calls, wl: Workload, steps: int, stream):
    """The same step through the public API with pinned host buffers: inputs
    are copied host -> device and results device -> host inside the timing."""
    torch = run.torch
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)  # noqa: E731
    if wl.name in ("multi", "multi_prefill"):
        h_in = [(pin(run.xs[0]), run.xs[0]), (pin(run.vid), run.vid)]
        h_out = [(pin(run.ys[0]), run.ys[0])]
    elif wl.name == "slice":
        h_in = [(pin(x), x) for x in run.xs] + [(pin(run.vid), run.vid)]
        h_out = [(pin(y), y) for y in run.ys]
    elif wl.name == "materialize":
        h_in = [(pin(run.wb), run.wb), (pin(run.signs[0]), run.signs[0]), (pin(run.alpha[0]), run.alpha[0])]
        h_out = [(pin(run.w_eff), run.w_eff)]
    elif wl.name == "monosoup":
        h_in = [(pin(run.wb), run.wb)] + [(pin(w), w) for w in run.wf] + [(pin(run.omega), run.omega)]
        h_out = [(pin(run.w_merged), run.w_merged)]
    elif wl.name == "prefill":
        h_in = [(pin(run.xs[0]), run.xs[0])]
        h_out = [(pin(run.ys[0]), run.ys[0])]
    else:
        h_in = [(pin(run.wb), run.wb), (pin(run.wf[0]), run.wf[0])] + [(pin(x), x) for x in run.xs]
        h_out = [(pin(run.signs[0]), run.signs[0]), (pin(run.alpha[0]), run.alpha[0])] + \
                [(pin(y), y) for y in run.ys]
    for h, d in h_in:
        h.copy_(d)
    h2d = sum(d.numel() * d.element_size() for _, d in h_in)
    d2h = sum(d.numel() * d.element_size() for _, d in h_out)

    def step():
        for h, d in h_in:
            d.copy_(h, non_blocking=True)
        for c in calls:
            c[4]()
        for h, d in h_out:
            h.copy_(d, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"value": None, "unit": "GB/s", "ms_per_step": ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "path": "pinned host -> device copies, bd_* calls, device -> host copies"}


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
