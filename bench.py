"""Benchmark of the BitDelta hot path on GB300.

Default workload (one GPU): the 70B-FFN-shaped decode GEMV -- W_base bf16
[28672 x 8192] ~ N(0, 0.02), Delta ~ Laplace(0, 1e-3), per-row alpha -- where
one step is the whole path over one batch: bd_compress (Delta, sign bits,
alpha) followed by the fused linear for 1, 4 and 16 tokens.  The metric is
HBM GB/s of algorithmic bytes per step; the JSON line also carries tokens/s,
the roofline of the dominant kernel (CUDA-event timed inside the timed
region), the CPU oracle timed on the host cores (all of them and one), an
end-to-end number with host buffers (the full step, and a serving step in
which the weights stay resident), and the SM clocks sampled during the timed
region.

The default line also carries one sub-measurement per other workload of the
serving setup, each timed in its own region with its own roofline, clocks
and CPU oracle baseline: "tiny" (256 x 256, T = 4, per-matrix alpha; L2-
resident, latency only), "multi" (8192 x 8192 shared W_base, 14 variants,
64 Zipf-routed tokens), "prefill" (4096 tokens x 8192 x 8192, tensor cores,
TFLOP/s) and "slice" (8 layers of a 70B-shaped stack, 56 multi-variant
linears, 14 variants compressed on the GPU, 32 decode tokens).  On one GPU it
also carries the rows past the serving setup: "materialize" (W_eff written
once, 28672 x 8192), "multi_prefill" (4096 Zipf-routed tokens over 14
variants, tensor cores) and "monosoup" (the merge of 3 task vectors of
8192 x 8192 at rank 16).

--workload runs any of them as the main line instead.  `python bench.py --impl reference` times the CPU oracle
instead (the reference arm), on bounded samples of the same workload.

Multi-GPU (--gpus N): one process per GPU.  Without a torchrun environment
the script relaunches itself under torch.distributed.run with N ranks.  Every
matrix is partitioned by output rows (rank r owns rows [r d_out / N,
(r + 1) d_out / N)); x is replicated; per-row alpha needs no exchange; a
per-matrix alpha takes one fp64 all-reduce; each rank's kernels read only
its own rows.  The timed region is bracketed by barriers and the slowest
rank's time is reported; value = the whole matrices' bytes / that time
(strong scaling).  The all-gather of y that a following layer would need is
timed separately ("exchange").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused BitDelta linear HBM GB/s (% of peak), tokens/s; prefill TFLOP/s (% peak)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DATA = "synthetic (seeded numpy / torch generators; shapes and distributions of the BitDelta serving setup)"

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch from
# one ncu capture (mean over the captured launches), keyed by kernel; each
# entry records the sha256 of the kernel's source file at capture time and is
# ignored once that source has changed.  Summaries of the captures are in profiles/.  An entry whose value
# is a float is a ratio (traffic / algorithmic bytes) taken on one launch of a
# smaller call of the same kernel and applied to the average launch.
MONOSOUP_CALL = "bd_monosoup_merge (tensor-core products, Gram / Cholesky / tridiagonal eigensolver, tensor-core merge)"
NCU_TRAFFIC = {
    # (kernel, workload): (source sha256[:16], source file, bytes per launch or ratio)
    ("skinny_kernel<1>", "decode"): ("0a72eed5c5ceea12", "bd_skinny.cu", 499_373_248 + 174_635),
    # 4 rows per CTA (kCompressRowsPerCta in bd_internal.h)
    ("compress_kernel", "decode"): ("75f8daf3ca961f7e", "bd_compress.cu", 939_559_381 + 6_489_301),
    ("prefill_kernel", "prefill"): ("4c65a422a15ad932", "bd_prefill.cu", 619_373_995 + 65_847_595),
    # multi_kernel only (the prepare pass adds about 3.7 MB of x tiles and corrections)
    ("multi_prepare + multi_kernel<8>", "multi"): ("a3057edfbaaadd8d", "bd_multi.cu", 255_719_211 + 114_603),
    # the grouped prefill_kernel only (router, plan and gather add about 134 MB of x copies)
    ("route + gather + prefill_kernel (grouped)", "multi_prefill"): ("4c65a422a15ad932", "bd_prefill.cu",
                                                                      939_384_576 + 60_230_955),
    ("materialize_kernel", "materialize"): ("62ad2eca0a51c12a", "bd_materialize.cu", 499_278_421 + 417_748_608),
    # all 26 launches of one merge (launch list with DRAM counters, one pass)
    (MONOSOUP_CALL, "monosoup"): ("da010de39fd26f35", "bd_monosoup.cu", 2_409_228_288 + 107_803_904),
}

# kernels each call launches: multi = prepare + fused kernel; multi_prefill =
# router + plan + gather + grouped prefill; monosoup = the merge's launches
LAUNCHES_PER_CALL = {"multi": 2, "slice": 2, "multi_prefill": 4, "monosoup": 26}
# workloads whose own figure is tensor throughput (TFLOP/s) rather than GB/s
TENSOR_WORKLOADS = ("prefill", "multi_prefill")
# the arithmetic type each workload computes in (the MonoSoup products and
# merge multiply exact three-piece bf16 splits of fp32 operands on the tensor
# cores with fp32 accumulation; Gram matrices and Cholesky factors in
# float-float)
DTYPES = {"monosoup": "bf16 pieces of fp32 (exact splits), f32 accumulate"}
# MonoSoup workload: k checkpoints, rank r, sketch width l, power iterations q
MONOSOUP = {"d": 8192, "k": 3, "rank": 16, "l": 32, "q": 1}
# sub-measurements of the default line: (name, timed steps, warm-up steps)
SUBS = (("tiny", 200, 10), ("multi", 20, 5), ("prefill", 20, 3), ("slice", 10, 3))
# the rows past the serving configurations (materialised variant, mixed-variant
# prefill, MonoSoup merge), measured in the default line on one GPU
SUBS_NEXT = (("materialize", 20, 3), ("multi_prefill", 20, 3), ("monosoup", 10, 3))
WORKLOADS = ("decode", "tiny", "multi", "prefill", "multi_prefill", "materialize", "monosoup", "slice")


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--workload", choices=WORKLOADS, default="decode")
    p.add_argument("--no-sub", action="store_true", help="skip the sub-measurements of the default line")
    p.add_argument("--sub", default="", help="comma-separated subset of the sub-measurements (default: all)")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    return p.parse_args(argv)


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


def row_span(d_out: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [r0, r1) of `rank` under the output-row partition (sizes differ by at most one)."""
    return d_out * rank // world, d_out * (rank + 1) // world


# ----------------------------------------------------------------------------- algorithmic bytes and FLOPs

def materialize_bytes(d_out, d_in, n_alpha):
    """W_base read, W_eff written (2 bytes each per weight), bits and alpha read."""
    return 4 * d_out * d_in + d_out * d_in // 8 + 4 * n_alpha


def monosoup_bytes(d, k, q):
    """Each of the 2 + 2q passes (sketch, 2q power-iteration products, B^T)
    reads every W_i and W_base once (the k products of a pass share the
    W_base tiles), plus the merge's W_base read and W_merged write."""
    return (2 + 2 * q) * (k + 1) * 2 * d * d + 4 * d * d


def monosoup_flops(d, k, rank, l, q):
    """Algorithmic FLOPs of the products with the task vectors (2 d^2 l each)
    and of the rank-(k r) merge (2 d^2 k r), counted once per product (the
    tensor cores multiply exact bf16 pieces of the fp32 operands, several
    piece products per algorithmic one)."""
    return k * (2 + 2 * q) * 2 * d * d * l + 2 * d * d * k * rank


def linear_bytes(T, d_out, d_in, n_alpha, y_bytes=2):
    """Algorithmic bytes of one fused linear: W_base + bits + alpha + x + y."""
    return 2 * d_out * d_in + d_out * d_in // 8 + 4 * n_alpha + 2 * T * d_in + y_bytes * T * d_out


def multi_bytes(T, d_out, d_in, n_active, per_row=True):
    """Multi-variant linear: W_base once + bits and alpha of every active
    variant + x + y + variant ids."""
    n_alpha = d_out if per_row else 1
    return 2 * d_out * d_in + n_active * (d_out * d_in // 8 + 4 * n_alpha) + 2 * T * d_in + 2 * T * d_out + 4 * T


def compress_bytes(d_out, d_in, n_alpha):
    """Algorithmic bytes of one compression: W_base + W_ft read, bits + alpha written."""
    return 4 * d_out * d_in + d_out * d_in // 8 + 4 * n_alpha


# ----------------------------------------------------------------------------- workloads

class Workload:
    """Host inputs (numpy bf16 bits) of one workload, restricted to the output
    rows [r0, r1) a rank owns (all rows for one GPU), plus its description."""

    def __init__(self, name, seed, world=1, rank=0):
        from bit_weight_delta_bd_gb300 import synth

        self.name, self.seed, self.world, self.rank = name, seed, world, rank
        self.wb, self.wf, self.xs, self.vid = None, [], [], None
        if name == "slice":  # weights are drawn on the device by SliceRun
            self.tokens = [32]
            self.per_row = True
            self.vid = synth.zipf_variant_ids(np.random.default_rng(seed), 32, 14)
            self.d_out_full = self.d_out = self.d_in = 0
            self.n_alpha = 0
            self.r0 = self.r1 = 0
            return
        if name in ("decode", "tiny"):
            d_out, d_in = (28672, 8192) if name == "decode" else (256, 256)
            self.tokens = [1, 4, 16] if name == "decode" else [4]
            self.per_row = name == "decode"
            rng = np.random.default_rng(seed)
            wb = synth.base_weight(rng, d_out, d_in)
            wfs = [synth.finetuned_weight(rng, wb, 1e-3)]
            self.xs = [synth.activations(rng, T, d_in) for T in self.tokens]
        elif name == "materialize":
            d_out, d_in = 28672, 8192
            self.tokens = []
            self.per_row = True
            wb, wf, _ = synth.single_problem(seed, d_out, d_in, 1)
            wfs = [wf]
        elif name == "monosoup":
            d_out = d_in = MONOSOUP["d"]
            self.tokens = []
            self.per_row = True
            wb, wfs = synth.monosoup_checkpoints(seed, d_out, d_in, MONOSOUP["k"], MONOSOUP["rank"])
            self.omega = synth.gaussian_test_matrix(seed + 1, d_in, MONOSOUP["l"])
        elif name == "prefill":
            d_out, d_in = 8192, 8192
            self.tokens = [4096]
            self.per_row = True
            wb, wf, x = synth.single_problem(seed + 3, d_out, d_in, 4096)
            wfs = [wf]
            self.xs = [x]
        else:  # multi (64 tokens, decode kernel) or multi_prefill (4096 tokens, tensor cores)
            d_out, d_in = 8192, 8192
            self.tokens = [4096 if name == "multi_prefill" else 64]
            self.per_row = True
            wb, wfs, x, self.vid, _ = synth.multi_problem(seed, d_out, d_in, self.tokens[0], 14)
            self.xs = [x]
        self.d_out_full, self.d_in = d_out, d_in
        if name == "monosoup" and world > 1:
            raise SystemExit("monosoup: the merge is not row-partitioned (its subspace spans every row); use --gpus 1")
        self.r0, self.r1 = row_span(d_out, world, rank)
        self.wb = np.ascontiguousarray(wb[self.r0:self.r1])
        self.wf = [np.ascontiguousarray(w[self.r0:self.r1]) for w in wfs]
        self.d_out = self.r1 - self.r0
        self.n_alpha = self.d_out if self.per_row else 1

    def active(self) -> int:
        return 0 if self.vid is None else len(set(int(v) for v in self.vid if v >= 0))

    def step_bytes_full(self) -> int:
        """Algorithmic bytes of one step over the whole matrices (all ranks' rows)."""
        return _step_bytes(self.name, self.d_out_full, self.d_in, self.tokens, self.per_row, self.active(),
                           len(self.wf))

    def step_flops_full(self) -> int:
        if self.name == "monosoup":
            return monosoup_flops(self.d_out_full, len(self.wf), MONOSOUP["rank"], MONOSOUP["l"], MONOSOUP["q"])
        if self.name == "slice":
            return sum(2 * 32 * d_out * d_in for _, d_out, d_in in _slice_linears()) * 8
        return sum(2 * T * self.d_out_full * self.d_in for T in self.tokens)

    def config(self):
        par = ("single GPU" if self.world == 1 else
               f"rows{self.world}: output rows of every matrix split over {self.world} GPUs, x replicated")
        if self.name == "slice":
            return {"workload": "slice_8_layers_70b_shapes_V14_T32", "layers": 8,
                    "linears": "q/o 8192x8192, k/v 8192->1024, gate/up 8192->28672, down 28672->8192",
                    "variants": 14, "active_variants": self.active(), "tokens": [32], "alpha": "per_row",
                    "step": "56 bd_linear_multi calls (variants compressed on the GPU once, untimed)",
                    "l2": "inputs larger than L2 (13.7 GB of W_base per step)", "parallelism": par}
        c = {"workload": self.name, "d_out": self.d_out_full, "d_in": self.d_in, "tokens": self.tokens,
             "alpha": "per_row" if self.per_row else "per_matrix"}
        if self.name == "decode":
            c["workload"] = "decode_ffn_28672x8192_T1_4_16"
            c["step"] = "bd_compress + bd_linear at T=1, 4, 16 (one variant)"
            c["l2"] = "inputs larger than L2 (W_base 470 MB, W_ft 470 MB vs 126.5 MB L2)"
        elif self.name == "prefill":
            c["workload"] = "prefill_4096x8192x8192"
            c["step"] = "bd_linear at T=4096, one variant (compressed once, untimed); tensor-core path"
            c["l2"] = "inputs larger than L2 (W_base 134 MB + x 67 MB + y 67 MB vs 126.5 MB L2)"
        elif self.name == "multi_prefill":
            c["workload"] = "multi_prefill_8192x8192_V14_T4096"
            c["variants"] = len(self.wf)
            c["active_variants"] = self.active()
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
            c["active_variants"] = self.active()
            c["step"] = "bd_linear_multi over 64 Zipf(1.1)-routed tokens (variants compressed once, untimed)"
            c["l2"] = "L2 flushed (256 MB write) before each step; flush excluded from kernel events"
        c["parallelism"] = par
        return c


def _slice_linears():
    from bit_weight_delta_bd_gb300 import synth

    return synth.SLICE_LINEARS


def _step_bytes(name, d_out, d_in, tokens, per_row, n_active, n_ckpt):
    n_alpha = d_out if per_row else 1
    if name == "slice":
        return 8 * sum(multi_bytes(32, o, i, n_active) for _, o, i in _slice_linears())
    if name in ("multi", "multi_prefill"):
        return multi_bytes(tokens[0], d_out, d_in, n_active, per_row)
    if name == "materialize":
        return materialize_bytes(d_out, d_in, n_alpha)
    if name == "monosoup":
        return monosoup_bytes(d_out, n_ckpt, MONOSOUP["q"])
    out = 0 if name == "prefill" else compress_bytes(d_out, d_in, n_alpha)
    return out + sum(linear_bytes(T, d_out, d_in, n_alpha) for T in tokens)


class DeviceRun:
    """Device copies of a workload (this rank's rows) and the calls of one step."""

    def __init__(self, wl: Workload, dev):
        import torch

        from bit_weight_delta_bd_gb300 import bitdelta as bd

        self.bd, self.torch, self.wl, self.dev = bd, torch, wl, dev
        self.mode = bd.BD_ALPHA_PER_ROW if wl.per_row else bd.BD_ALPHA_PER_MATRIX
        rows, d_in = max(wl.d_out, 0), wl.d_in

        def d(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

        self.wb = d(wl.wb)
        self.wf = [d(w) for w in wl.wf]
        self.xs = [d(x) for x in wl.xs]
        self.signs = [torch.empty((rows, d_in // 32), dtype=torch.int32, device=dev) for _ in wl.wf]
        self.alpha = [torch.full((wl.n_alpha,), float("nan"), dtype=torch.float32, device=dev) for _ in wl.wf]
        self.ys = [torch.empty((T, rows), dtype=torch.bfloat16, device=dev) for T in wl.tokens]
        self.ws = bd.new_workspace(max(bd.bd_compress_workspace_size(rows, d_in, self.mode),
                                       bd.bd_linear_workspace_size(64, rows, d_in),
                                       bd.bd_linear_multi_workspace_size(max(64, max(wl.tokens, default=0)),
                                                                         max(len(wl.wf), 1), rows, d_in)), dev)
        self.vid = None if wl.vid is None else torch.from_numpy(wl.vid).to(dev)
        self.flush = None
        self.alpha_exchange = None  # per-matrix alpha over row partitions: the one collective of a step
        if wl.name == "materialize":
            self.w_eff = torch.empty((rows, d_in), dtype=torch.int16, device=dev)
        if wl.name == "monosoup":
            self.omega = torch.from_numpy(wl.omega).to(dev)
            self.w_merged = torch.empty((rows, d_in), dtype=torch.bfloat16, device=dev)
            self.ws_ms = bd.new_workspace(bd.bd_monosoup_workspace_size(rows, d_in, len(wl.wf),
                                                                        MONOSOUP["rank"], MONOSOUP["l"]), dev)
        if wl.name in ("multi", "prefill", "multi_prefill", "materialize"):
            for v in range(len(wl.wf)):  # variants are compressed once, before timing
                bd.bd_compress(self.wb, self.wf[v], self.mode, self.signs[v], self.alpha[v], self.ws)
            torch.cuda.synchronize()
            self.wf = []  # W_ft is not needed any more
            torch.cuda.empty_cache()
        if wl.name == "multi":
            self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        if wl.world > 1 and not wl.per_row:
            from bit_weight_delta_bd_gb300 import shard

            def exchange():
                a = shard.per_matrix_alpha_allreduce(self.alpha[0].cpu() if _backend() == "gloo" else self.alpha[0],
                                                     wl.d_out, wl.d_out_full)
                self.alpha[0].copy_(a)
            self.alpha_exchange = exchange

    def calls(self):
        """[(label, kernel name, algorithmic bytes (this rank), flops, fn)] of one step."""
        bd, wl = self.bd, self.wl
        out = []
        if wl.name in ("multi", "multi_prefill"):
            T = wl.tokens[0]
            nbytes = multi_bytes(T, wl.d_out, wl.d_in, wl.active(), wl.per_row)
            kname = ("route + gather + prefill_kernel (grouped)" if wl.name == "multi_prefill"
                     else "multi_prepare + multi_kernel<8>")
            flops = 2 * T * wl.d_out * wl.d_in
            out.append((f"linear_multi_T{T}", kname, nbytes, flops,
                        lambda: bd.bd_linear_multi(self.xs[0], self.vid, self.signs, self.alpha, self.mode, self.wb,
                                                   self.ys[0], self.ws)))
            return out
        if wl.name == "monosoup":
            m = MONOSOUP
            out.append(("monosoup_merge", MONOSOUP_CALL,
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

        def compress():
            bd.bd_compress(self.wb, self.wf[0], self.mode, self.signs[0], self.alpha[0], self.ws)
            if self.alpha_exchange is not None:
                self.alpha_exchange()
        out.append(("compress", "compress_kernel", compress_bytes(wl.d_out, wl.d_in, wl.n_alpha), 0, compress))
        for i, T in enumerate(wl.tokens):
            nt = 1 if T <= 8 else 2 if T <= 16 else 4 if T <= 32 else 8
            out.append((f"linear_T{T}", f"skinny_kernel<{nt}>", linear_bytes(T, wl.d_out, wl.d_in, wl.n_alpha),
                        2 * T * wl.d_out * wl.d_in,
                        (lambda i=i: bd.bd_linear(self.xs[i], self.wb, self.signs[0], self.alpha[0], self.mode,
                                                  self.ys[i], self.ws))))
        return out

    def serving_calls(self):
        """The linears alone (weights, signs and alpha resident): the steady-state serving step."""
        return [c for c in self.calls() if c[0] != "compress"]


class SliceRun:
    """The 8-layer slice resident on the device: per linear W_base and the 14
    variants' packed signs and alpha (compressed here, on the GPU, from
    on-device seeded draws), plus that linear's 32-token input.  With
    world > 1 each matrix keeps only this rank's rows.  `sample_rows` rows of
    every matrix are also kept on the host (W_base and every W_ft) for the
    CPU oracle baseline."""

    def __init__(self, wl: Workload, dev, seed: int, layers: int = 8, sample_rows: int = 0):
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
        self.mats, self.samples = [], []
        for layer in range(layers):
            for m, (name, d_out, d_in) in enumerate(synth.SLICE_LINEARS):
                r0, r1 = row_span(d_out, wl.world, wl.rank)
                wb_full = synth.device_base_weight(synth.slice_seed(seed, layer, m), d_out, d_in, dev)
                wb = wb_full[r0:r1].contiguous()
                smp = None
                if sample_rows:
                    rows = synth.sample_rows(layer * 7 + m, r1 - r0, sample_rows)
                    ridx = torch.from_numpy(rows + r0).to(dev)
                    smp = {"rows": rows, "d_out": r1 - r0, "d_in": d_in, "wb": _bits16(wb_full[ridx]), "wf": []}
                signs, alphas = [], []
                for v in range(V):
                    wf_full = synth.device_finetuned_weight(synth.slice_seed(seed, layer, m, v), wb_full,
                                                            float(scales[v]))
                    wf = wf_full[r0:r1].contiguous()
                    if smp is not None:
                        smp["wf"].append(_bits16(wf_full[ridx]))
                    del wf_full
                    sg = torch.empty((r1 - r0, d_in // 32), dtype=torch.int32, device=dev)
                    al = torch.empty(r1 - r0, dtype=torch.float32, device=dev)
                    bd.bd_compress(wb, wf, bd.BD_ALPHA_PER_ROW, sg, al, self.ws)
                    del wf
                    signs.append(sg)
                    alphas.append(al)
                del wb_full
                x_host = synth.activations(rng, T, d_in)
                x = torch.from_numpy(x_host.view(np.int16)).to(dev)
                y = torch.empty((T, r1 - r0), dtype=torch.bfloat16, device=dev)
                self.mats.append((f"L{layer}.{name}", r1 - r0, d_in, wb, signs, alphas, x, y))
                if smp is not None:
                    smp["x"] = x_host
                    self.samples.append(smp)
        torch.cuda.synchronize()
        if bd.bd_check_async(self.ws) != bd.BD_OK:
            raise RuntimeError("asynchronous error while compressing the slice")
        self.flush = None
        self.alpha_exchange = None
        self.xs = [mt[6] for mt in self.mats]
        self.ys = [mt[7] for mt in self.mats]

    def calls(self):
        bd, wl = self.bd, self.wl
        active = wl.active()
        T = 32
        out = []
        for label, d_out, d_in, wb, signs, alphas, x, y in self.mats:
            out.append((label, "multi_prepare + multi_kernel<4>", multi_bytes(T, d_out, d_in, active),
                        2 * T * d_out * d_in,
                        (lambda wb=wb, signs=signs, alphas=alphas, x=x, y=y:
                         bd.bd_linear_multi(x, self.vid, signs, alphas, bd.BD_ALPHA_PER_ROW, wb, y, self.ws))))
        return out

    def serving_calls(self):
        return self.calls()


def _bits16(t) -> np.ndarray:
    return t.contiguous().view(__import__("torch").int16).cpu().numpy().view(np.uint16)


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

def _cpu_cores() -> int:
    return os.cpu_count() or 1


def oracle_time(wl: Workload, budget_s: float = 12.0, threads: int = 0, slice_samples=None):
    """Times the CPU oracle (as it stands) on a bounded sample of one step:
    whole steps for a small matrix, growing row blocks of one step for a large
    one, until `budget_s` of wall time is spent.  Work the GPU step does not
    time (compressing variants that are resident before the step) is done
    before the clock starts.  Returns (GB/s of algorithmic bytes, threads
    used, sample description)."""
    import oracle

    cores = oracle.set_threads(threads if threads > 0 else _cpu_cores())
    step_bytes = wl.step_bytes_full()
    if wl.name == "slice":
        return _oracle_time_slice(wl, slice_samples, cores, step_bytes)
    d_out, d_in = wl.d_out, wl.d_in
    scale = wl.d_out_full / max(d_out, 1)  # this rank's rows stand for the whole matrices
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
    compress_in_step = wl.name in ("decode", "tiny")
    if d_out * d_in <= (1 << 20):  # small: whole steps
        n, t_used = 0, 0.0
        while t_used < budget_s or n == 0:
            t0 = time.perf_counter()
            s, a = oracle.compress(wl.wb, wl.wf[0], wl.per_row)
            for x in wl.xs:
                oracle.linear(x, wl.wb, s, a, wl.per_row)
            t_used += time.perf_counter() - t0
            n += 1
        return step_bytes * n / (t_used * scale) / 1e9, cores, f"{n} whole steps ({t_used:.2f} s on {cores} threads)"
    rows_done, t_used, chunk = 0, 0.0, 16
    while (t_used < budget_s or rows_done == 0) and rows_done < d_out:
        r = np.arange(rows_done, min(d_out, rows_done + chunk), dtype=np.int64)
        t_prep = time.perf_counter()
        sfs, afs = [], []
        for wf in wl.wf:
            s, a = oracle.compress_rows(wl.wb, wf, r)
            sf = np.zeros((d_out, d_in // 32), np.uint32)
            af = np.zeros(d_out, np.float32)
            sf[r], af[r] = s, a
            sfs.append(sf)
            afs.append(af)
        t0 = time.perf_counter()
        if wl.name == "materialize":
            oracle.materialize(wl.wb[r], sfs[0][r], afs[0][r], True)
        elif wl.vid is None:
            for x in wl.xs:
                oracle.linear(x, wl.wb, sfs[0], afs[0], True, rows=r)
        else:
            oracle.linear_multi(wl.xs[0], wl.vid, sfs, afs, True, wl.wb, rows=r)
        t_end = time.perf_counter()
        t_used += t_end - (t_prep if compress_in_step else t0)
        rows_done += len(r)
        chunk = min(chunk * 2, 4096)
    gbs = step_bytes * rows_done / (d_out * scale) / t_used / 1e9
    what = "compression and linears" if compress_in_step else "linears (variants compressed before the clock)"
    sample = f"{rows_done} of {d_out} rows of one step, {what} ({t_used:.2f} s on {cores} threads)"
    return gbs, cores, sample


def _oracle_time_slice(wl: Workload, samples, cores: int, step_bytes: int):
    """The slice step on the CPU: for every one of the 56 linears, the oracle
    multi-variant linear of the 32 tokens over a seeded sample of its rows
    (W_base and each variant's W_ft rows drawn by the same generators as the
    GPU's inputs, compressed by the oracle before the clock starts); the time
    of each linear is scaled by its rows / sampled rows."""
    import oracle

    if not samples:
        raise RuntimeError("the slice CPU baseline needs the sampled rows")
    t_full, t_used, n_rows = 0.0, 0.0, 0
    vid = wl.vid
    for smp in samples:
        loc = np.arange(len(smp["rows"]), dtype=np.int64)
        refs = [oracle.compress_rows(smp["wb"], wf, loc) for wf in smp["wf"]]
        t0 = time.perf_counter()
        oracle.linear_multi(smp["x"], vid, [r[0] for r in refs], [r[1] for r in refs], True, smp["wb"])
        dt = time.perf_counter() - t0
        t_used += dt
        n_rows += len(loc)
        t_full += dt * smp["d_out"] / len(loc)
    total_rows = sum(s["d_out"] for s in samples)
    t_full *= wl.world  # this rank's rows stand for the whole matrices
    return (step_bytes / t_full / 1e9, cores,
            f"{n_rows} of {total_rows} rows (a seeded sample of every one of the {len(samples)} linears; "
            f"{t_used:.2f} s on {cores} threads), scaled per linear to a full step ({t_full:.1f} s)")


def cpu_baseline(wl: Workload, unit: str, budget_s: float = 10.0, slice_samples=None) -> dict:
    """The oracle on all host cores and on one core, in the line's unit."""
    out = {}
    for key, thr in (("all", 0), ("one", 1)):
        gbs, cores, sample = oracle_time(wl, budget_s=budget_s if thr == 0 else budget_s / 2, threads=thr,
                                         slice_samples=slice_samples)
        value = gbs
        if unit == "TFLOP/s":
            value = wl.step_flops_full() / (wl.step_bytes_full() / (gbs * 1e9)) / 1e12
        elif unit == "tokens/s":
            value = sum(wl.tokens) / (wl.step_bytes_full() / (gbs * 1e9))
        out[key] = {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample}
    import oracle

    oracle.set_threads(_cpu_cores())
    line = dict(out["all"])
    line["single_thread"] = {k: out["one"][k] for k in ("value", "cores", "sample")}
    return line


# ----------------------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _backend() -> str:
    import torch.distributed as dist

    return dist.get_backend() if dist.is_initialized() else "none"


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def spawn_ranks(n: int, argv) -> int:
    """Relaunches this script under torch.distributed.run with n ranks on
    this node (127.0.0.1 rendezvous) and returns its exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.abspath(__file__), *argv]
    return subprocess.run(cmd, cwd=ROOT).returncode


def gather_rows(y_local, d_out: int, world: int, rank: int, group=None):
    """All-gather of a row-partitioned output: y_local [T][rows of `rank`]
    -> y [T][d_out] on every rank (shards padded to the largest row count,
    so that every rank sends one equal-sized buffer)."""
    import torch
    import torch.distributed as dist

    spans = [row_span(d_out, world, r) for r in range(world)]
    width = max(b - a for a, b in spans)
    T = y_local.shape[0]
    send = torch.zeros((width, T), dtype=y_local.dtype, device=y_local.device)
    send[:y_local.shape[1]] = y_local.t()
    recv = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(recv, send, group=group)
    return torch.cat([recv[r][:b - a] for r, (a, b) in enumerate(spans)], dim=0).t().contiguous()


def _max_over_ranks(v: float, dev, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device=dev if _backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ----------------------------------------------------------------------------- timing

def time_steps(run, calls, steps: int, warmup: int, world: int, dev, local: int):
    """W warm-up steps, then exactly `steps` timed steps bracketed by a barrier
    and a device synchronize on both sides, CUDA events around every call on
    the launching stream, clocks sampled during the region.  Returns
    (ms per step of this rank, per-call event times [steps][calls] in ms,
    clock summary)."""
    import torch

    stream = torch.cuda.current_stream()

    def one_step(evs=None):
        if run.flush is not None:
            run.flush.fill_(1)
        for i, c in enumerate(calls):
            if evs is not None:
                evs[i][0].record(stream)
            c[4]()
            if evs is not None:
                evs[i][1].record(stream)

    for _ in range(max(warmup, 3)):
        one_step()
    if run.bd.bd_check_async(run.ws) != run.bd.BD_OK:
        raise RuntimeError("asynchronous error during warm-up")
    torch.cuda.synchronize()
    events = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in calls]
              for _ in range(steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(_smi_id(local))
    t_start.record(stream)
    for k in range(steps):
        one_step(events[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    clk = clocks.stop()
    if run.bd.bd_check_async(run.ws) != run.bd.BD_OK:
        raise RuntimeError("asynchronous error during the timed region")
    ev_ms = [[events[k][i][0].elapsed_time(events[k][i][1]) for i in range(len(calls))] for k in range(steps)]
    elapsed = t_start.elapsed_time(t_end)
    if run.flush is not None:  # the L2 flush is not part of the path: count kernel time only
        elapsed = sum(sum(r) for r in ev_ms)
    return elapsed / steps, ev_ms, clk


def roofline_of(wl: Workload, calls, ev_ms, hbm_peak, bf16_peak, peak_src):
    """Roofline of the dominant kernel (largest share of the events' time):
    achieved = algorithmic bytes (or FLOPs) per launch / its average
    CUDA-event duration; plus the per-kernel table."""
    per_kernel = {}
    for i, (label, kname, nbytes, flops, _) in enumerate(calls):
        ms = [row[i] for row in ev_ms]
        e = per_kernel.setdefault(kname, {"launches": 0, "total_ms": 0.0, "bytes": 0, "flops": 0, "labels": []})
        e["launches"] += len(ms)
        e["total_ms"] += sum(ms)
        e["bytes"] += nbytes * len(ms)
        e["flops"] += flops * len(ms)
        e["labels"].append(label)
    dom = max(per_kernel, key=lambda k: per_kernel[k]["total_ms"])
    d = per_kernel[dom]
    avg_ms = d["total_ms"] / d["launches"]
    bytes_per_launch = d["bytes"] / d["launches"]
    flops_per_launch = d["flops"] / d["launches"]
    achieved = bytes_per_launch / (avg_ms * 1e-3) / 1e9
    traffic = None
    tr = NCU_TRAFFIC.get((dom, wl.name))
    if tr is not None and tr[0] == _src_sha(tr[1]) and wl.world == 1:
        traffic = tr[2] * bytes_per_launch if isinstance(tr[2], float) else tr[2]
    if wl.name in TENSOR_WORKLOADS:
        tf = flops_per_launch / (avg_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": tf / bf16_peak, "traffic": traffic, "peak_source": f"{peak_src} (bf16_tflops, burst)",
                "flops_per_launch": flops_per_launch, "avg_launch_us": avg_ms * 1e3}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": traffic, "peak_source": f"{peak_src} (hbm_gbs)",
                "bytes_per_launch": bytes_per_launch, "avg_launch_us": avg_ms * 1e3}
    tot = sum(x["total_ms"] for x in per_kernel.values())
    kernels = {k: {"launches": v["launches"], "avg_us": v["total_ms"] / v["launches"] * 1e3,
                   "share": v["total_ms"] / tot, "GBps": v["bytes"] / (v["total_ms"] * 1e-3) / 1e9,
                   "frac_hbm": v["bytes"] / (v["total_ms"] * 1e-3) / 1e9 / hbm_peak,
                   "calls": v["labels"] if len(v["labels"]) <= 4 else f"{len(v['labels'])} calls"}
               for k, v in per_kernel.items()}
    return roof, kernels


def _unit_of(name: str) -> str:
    return "TFLOP/s" if name in TENSOR_WORKLOADS else "GB/s"


def _value(wl: Workload, ms_per_step: float) -> float:
    """Whole-job figure of one step that took ms_per_step (all ranks' rows)."""
    if _unit_of(wl.name) == "TFLOP/s":
        return wl.step_flops_full() / (ms_per_step * 1e-3) / 1e12
    return wl.step_bytes_full() / (ms_per_step * 1e-3) / 1e9


def make_run(wl: Workload, dev, sample_rows: int = 0):
    if wl.name == "slice":
        return SliceRun(wl, dev, wl.seed, sample_rows=sample_rows)
    return DeviceRun(wl, dev)


def measure(name, args, steps, warmup, world, rank, local, dev, peaks, want_cpu):
    """One workload in its own timed region: the line fields for it."""
    import torch

    hbm_peak, bf16_peak, peak_src = peaks
    wl = Workload(name, args.seed, world, rank)
    run = make_run(wl, dev, sample_rows=128 if (want_cpu and rank == 0) else 0)
    calls = run.calls()
    ms_local, ev_ms, clk = time_steps(run, calls, steps, warmup, world, dev, local)
    ms = _max_over_ranks(ms_local, dev, world)
    roof, kernels = roofline_of(wl, calls, ev_ms, hbm_peak, bf16_peak, peak_src)
    unit = _unit_of(name)
    out = {"workload": wl.config()["workload"], "config": wl.config(), "value": _value(wl, ms), "unit": unit,
           "ms_per_step": ms, "steps": steps, "warmup": warmup,
           "tokens_per_s": sum(wl.tokens) / (ms * 1e-3) if wl.tokens else None,
           "roofline": roof, "kernels": kernels, "clocks": clk,
           "gpu_launches": LAUNCHES_PER_CALL.get(name, 1) * len(calls) * steps + (steps if not wl.per_row else 0)}
    if name == "tiny":
        out["roofline"] = None  # 139 KB stay in L2: latency only
        out["latency_us"] = ms * 1e3
        out["kernels"] = kernels
    out["cpu_baseline"] = None
    if want_cpu and rank == 0:
        out["cpu_baseline"] = cpu_baseline(wl, unit, slice_samples=getattr(run, "samples", None))
    del run
    torch.cuda.empty_cache()
    return out


def measure_exchange(run, wl: Workload, dev, world: int, reps: int = 20):
    """The all-gather of every linear's y that a following layer would need
    (row-partitioned outputs to full rows on every rank), timed on its own."""
    import torch

    if world == 1 or not getattr(run, "ys", None):
        return None
    full = [wl.d_out_full] * len(run.ys) if wl.name != "slice" else [None] * len(run.ys)
    if wl.name == "slice":
        full = [d for _ in range(8) for _, d, _ in _slice_linears()]

    def step():
        for y, d_out in zip(run.ys, full):
            gather_rows(y, d_out, world, wl.rank)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    _barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        step()
    b.record()
    torch.cuda.synchronize()
    ms = _max_over_ranks(a.elapsed_time(b) / reps, dev, world)
    nbytes = sum(y.shape[0] * d * y.element_size() for y, d in zip(run.ys, full))
    return {"collective": "all_gather of y per linear (NCCL)", "ms_per_step": ms, "bytes_per_step": nbytes,
            "GBps": nbytes / (ms * 1e-3) / 1e9}


# ----------------------------------------------------------------------------- arms

def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    wl = Workload(args.workload, args.seed, world, 0)
    unit = _unit_of(wl.name)
    slice_samples = None
    if wl.name == "slice":
        import torch

        if not torch.cuda.is_available():
            print(json.dumps({"impl": "reference", "unavailable": "the slice inputs are drawn by torch's CUDA "
                              "generator; no GPU here to draw them"}), flush=True)
            return 0
        slice_samples = SliceRun(wl, torch.device("cuda", 0), args.seed, sample_rows=128).samples
    # each step is a bounded sample so that the whole run stays near 90 s of oracle time
    budget = max(0.01, min(12.0, 90.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        oracle_time(wl, budget_s=budget / 4, slice_samples=slice_samples)
    vals = []
    cores, sample = 0, ""
    for _ in range(args.steps):
        gbs, cores, sample = oracle_time(wl, budget_s=budget, slice_samples=slice_samples)
        vals.append(gbs)
    gbs = statistics.median(vals)
    ms_per_step = wl.step_bytes_full() / (gbs * 1e9) * 1e3
    value = _value(wl, ms_per_step)
    line = {"metric": METRIC, "value": value, "unit": unit, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "strong" if world > 1 else "weak", "vs_baseline": None,
            "dtype": "f64", "data": DATA, "config": wl.config(),
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

    if rank == 0:
        __graft_entry__.build()
    _barrier(world)
    __graft_entry__.build()  # no-op once built; loads the library on every rank
    peaks = load_peaks()
    hbm_peak, bf16_peak, peak_src = peaks

    wl = Workload(args.workload, args.seed, world, rank)
    run = make_run(wl, dev, sample_rows=128 if (rank == 0 and not args.no_cpu) else 0)
    calls = run.calls()
    ms_local, ev_ms, clk = time_steps(run, calls, args.steps, args.warmup, world, dev, local)
    ms_per_step = _max_over_ranks(ms_local, dev, world)
    roofline, kernels = roofline_of(wl, calls, ev_ms, hbm_peak, bf16_peak, peak_src)
    unit = _unit_of(wl.name)
    value = _value(wl, ms_per_step)
    step_bytes = wl.step_bytes_full()

    e2e = e2e_serving = None
    if not args.no_e2e:
        e2e = run_e2e(run, calls, wl, max(3, min(args.steps, 20)), world, dev)
        if wl.name in ("decode", "tiny"):
            e2e_serving = run_e2e(run, run.serving_calls(), wl, max(3, min(args.steps, 20)), world, dev,
                                  serving=True)
    exchange = measure_exchange(run, wl, dev, world)
    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(wl, unit, budget_s=12.0, slice_samples=getattr(run, "samples", None))
    launches = LAUNCHES_PER_CALL.get(wl.name, 1) * len(calls) * args.steps
    if not wl.per_row:
        launches += args.steps  # the per-matrix alpha's finalize pass
    del run, calls
    torch.cuda.empty_cache()

    subs = {}
    if wl.name == "decode" and not args.no_sub:
        subs_all = SUBS + (SUBS_NEXT if world == 1 else ())
        want = [s for s in args.sub.split(",") if s] or [s[0] for s in subs_all]
        for name, steps, warmup in subs_all:
            if name in want:
                subs[name] = measure(name, args, steps, warmup, world, rank, local, dev, peaks,
                                     want_cpu=not args.no_cpu)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "strong" if world > 1 else "weak", "vs_baseline": None,
                "dtype": DTYPES.get(wl.name, "bf16"), "accumulate": "f32", "data": DATA,
                "config": wl.config(),
                "tokens_per_s": sum(wl.tokens) / (ms_per_step * 1e-3) if wl.tokens else None,
                "frac_hbm_step": step_bytes / (ms_per_step * 1e-3) / 1e9 / world / hbm_peak,
                "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
                "e2e_serving": e2e_serving, "exchange": exchange, "clocks": clk, "gpu_launches": launches}
        line.update(subs)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(run, calls, wl: Workload, steps: int, world: int, dev, serving: bool = False):
    """The same step through the public API with pinned host buffers: this
    step's inputs are copied host -> device and its results device -> host
    inside the timing.  serving=True: the steady-state serving step, in which
    W_base, the signs and alpha stay resident and only x and y cross."""
    torch = run.torch
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)  # noqa: E731
    if serving or wl.name in ("multi", "multi_prefill", "prefill", "slice"):
        h_in = [(pin(x), x) for x in run.xs] + ([(pin(run.vid), run.vid)] if run.vid is not None else [])
        h_out = [(pin(y), y) for y in run.ys]
    elif wl.name == "materialize":
        h_in = [(pin(run.wb), run.wb), (pin(run.signs[0]), run.signs[0]), (pin(run.alpha[0]), run.alpha[0])]
        h_out = [(pin(run.w_eff), run.w_eff)]
    elif wl.name == "monosoup":
        h_in = [(pin(run.wb), run.wb)] + [(pin(w), w) for w in run.wf] + [(pin(run.omega), run.omega)]
        h_out = [(pin(run.w_merged), run.w_merged)]
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
    _barrier(world)
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = _max_over_ranks(a.elapsed_time(b) / steps, dev, world)
    if serving:
        nbytes = world * sum(c[2] for c in calls)
        if world > 1:
            nbytes = sum(linear_bytes(T, wl.d_out_full, wl.d_in, wl.d_out_full if wl.per_row else 1)
                         for T in wl.tokens)
        unit, value = "GB/s", nbytes / (ms * 1e-3) / 1e9
        path = ("pinned host -> device copies of x, bd_linear calls on resident W_base / signs / alpha, "
                "device -> host copies of y")
    else:
        unit = _unit_of(wl.name)
        value = _value(wl, ms)
        path = "pinned host -> device copies, bd_* calls, device -> host copies"
    out = {"value": value, "unit": unit, "ms_per_step": ms, "h2d_bytes_per_step": h2d * world,
           "d2h_bytes_per_step": d2h * world, "steps": steps, "path": path}
    if serving:
        out["tokens_per_s"] = sum(wl.tokens) / (ms * 1e-3)
    return out


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    args = parse_args(argv)
    if args.gpus < 1:
        raise SystemExit("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return spawn_ranks(args.gpus, argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but the launcher started {world} ranks (WORLD_SIZE)")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
