"""Runs every compute entry point of the library once per case on cuda:0 and
saves each output to an .npz file, for the bounds-checked build's test: the
test runs this script twice, as a child process with BD_LIBRARY naming the
normal library and then the bounds-checked one, and compares the two files.

Usage: python tests/bounds_run.py OUT.npz

The cases cover every kernel: compression (both alpha modes, the
no-allocation entry), the decode kernel at T = 1, 4, 16 and 64, the prefill
kernel at T = 100 and 600, multi-variant decode and prefill (base-model
tokens included), routing, materialisation, the fp32 reconstruction and the
MonoSoup merge on both of its product paths (l <= 32 on tensor cores, l > 32
on CUDA cores) with bf16 and fp32 outputs.  The last line printed is a JSON
object with the bounds status, the kernel bits and whether the loaded
library is the bounds-checked build.
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from bit_weight_delta_bd_gb300 import bitdelta as bd  # noqa: E402
from bit_weight_delta_bd_gb300 import synth  # noqa: E402


def _d(a: np.ndarray, dev) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(dev)
    return torch.from_numpy(a).to(dev)


def _h(t: torch.Tensor) -> np.ndarray:
    """Host copy as raw bits (bf16 as uint16, fp32 as uint32), so that the
    comparison is bitwise."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.int16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float32, torch.int32):
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.numpy()


def run(out_path: str) -> dict:
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    res: dict[str, np.ndarray] = {}
    d_out, d_in = 1000, 1024

    # compression, both alpha modes, workspace and no-allocation entries
    wb, wf, _ = synth.single_problem(11, d_out, d_in, 1)
    wb_d, wf_d = _d(wb, dev), _d(wf, dev)
    packed = {}
    for mode in (bd.BD_ALPHA_PER_MATRIX, bd.BD_ALPHA_PER_ROW):
        n_a = d_out if mode == bd.BD_ALPHA_PER_ROW else 1
        s = torch.zeros((d_out, d_in // 32), dtype=torch.int32, device=dev)
        a = torch.zeros(n_a, dtype=torch.float32, device=dev)
        ws = bd.new_workspace(bd.bd_compress_workspace_size(d_out, d_in, mode), dev)
        bd.bd_compress(wb_d, wf_d, mode, s, a, ws)
        assert bd.bd_check_async(ws) == bd.BD_OK
        res[f"compress_s_{mode}"], res[f"compress_a_{mode}"] = _h(s), _h(a)
        packed[mode] = (s, a)
        s2 = torch.zeros_like(s)
        a2 = torch.zeros_like(a)
        bd.bd_compress_noalloc(wb_d, wf_d, mode, s2, a2)
        res[f"noalloc_s_{mode}"], res[f"noalloc_a_{mode}"] = _h(s2), _h(a2)

    # single-variant linear: decode (T <= 64) and prefill (T > 64), both output types
    for T in (1, 4, 16, 64, 100, 600):
        x = _d(synth.activations(np.random.default_rng(100 + T), T, d_in), dev)
        for mode, (s, a) in packed.items():
            for odt in (torch.bfloat16, torch.float32):
                y = torch.zeros((T, d_out), dtype=odt, device=dev)
                ws = bd.new_workspace(bd.bd_linear_workspace_size(T, d_out, d_in), dev)
                bd.bd_linear(x, wb_d, s, a, mode, y, ws)
                assert bd.bd_check_async(ws) == bd.BD_OK
                res[f"linear_T{T}_m{mode}_{str(odt)[6:]}"] = _h(y)

    # multi-variant linear, per-row alpha, with base-model tokens (vid = -1)
    V, dm_out = 5, 776
    wbm, wfs, _, _, _ = synth.multi_problem(21, dm_out, d_in, 1, V)
    wbm_d = _d(wbm, dev)
    s_list, a_list = [], []
    for v in range(V):
        s = torch.zeros((dm_out, d_in // 32), dtype=torch.int32, device=dev)
        a = torch.zeros(dm_out, dtype=torch.float32, device=dev)
        ws = bd.new_workspace(bd.bd_compress_workspace_size(dm_out, d_in, bd.BD_ALPHA_PER_ROW), dev)
        bd.bd_compress(wbm_d, _d(wfs[v], dev), bd.BD_ALPHA_PER_ROW, s, a, ws)
        s_list.append(s)
        a_list.append(a)
    for T in (1, 7, 16, 64, 300, 700):
        rng = np.random.default_rng(200 + T)
        x = _d(synth.activations(rng, T, d_in), dev)
        vid_h = synth.zipf_variant_ids(rng, T, V).astype(np.int32)
        vid_h[::5] = -1
        vid = _d(vid_h, dev)
        for odt in (torch.bfloat16, torch.float32):
            y = torch.zeros((T, dm_out), dtype=odt, device=dev)
            ws = bd.new_workspace(bd.bd_linear_multi_workspace_size(T, V, dm_out, d_in), dev)
            bd.bd_linear_multi(x, vid, s_list, a_list, bd.BD_ALPHA_PER_ROW, wbm_d, y, ws)
            assert bd.bd_check_async(ws) == bd.BD_OK
            res[f"multi_T{T}_{str(odt)[6:]}"] = _h(y)

    # routing alone
    T, V = 3001, 14
    vid_h = synth.zipf_variant_ids(np.random.default_rng(31), T, V).astype(np.int32)
    vid_h[::7] = -1
    perm = torch.zeros(T, dtype=torch.int32, device=dev)
    seg = torch.zeros(V + 2, dtype=torch.int32, device=dev)
    ws = bd.new_workspace(bd.bd_route_workspace_size(T, V), dev)
    bd.bd_route(_d(vid_h, dev), V, perm, seg, ws)
    assert bd.bd_check_async(ws) == bd.BD_OK
    res["route_perm"], res["route_seg"] = _h(perm), _h(seg)

    # materialisation and the fp32 reconstruction
    for mode, (s, a) in packed.items():
        w = torch.zeros((d_out, d_in), dtype=torch.bfloat16, device=dev)
        bd.bd_materialize(wb_d, s, a, mode, w)
        res[f"materialize_{mode}"] = _h(w)
        w32 = torch.zeros((d_out, d_in), dtype=torch.float32, device=dev)
        bd.bd_debug_reconstruct(wb_d, s, a, mode, w32)
        res[f"reconstruct_{mode}"] = _h(w32)

    # MonoSoup merge: tensor-core products (l <= 32) and CUDA-core products (l > 32)
    for (mo, mi, k, r, l, q) in ((256, 384, 3, 4, 16, 1), (300, 256, 3, 8, 48, 1), (200, 256, 5, 6, 32, 2)):
        mwb, mws = synth.monosoup_checkpoints(41 + l, mo, mi, k, r)
        om = _d(synth.gaussian_test_matrix(51 + l, mi, l), dev)
        mwb_d = _d(mwb, dev)
        mws_d = [_d(w, dev) for w in mws]
        for odt in (torch.bfloat16, torch.float32):
            out = torch.zeros((mo, mi), dtype=odt, device=dev)
            ws = bd.new_workspace(bd.bd_monosoup_workspace_size(mo, mi, k, r, l), dev)
            bd.bd_monosoup_merge(mwb_d, mws_d, r, l, q, om, out, ws)
            assert bd.bd_check_async(ws) == bd.BD_OK
            res[f"monosoup_{mo}x{mi}_k{k}_l{l}_{str(odt)[6:]}"] = _h(out)

    torch.cuda.synchronize()
    st, bits = bd.bd_debug_bounds_check()
    np.savez(out_path, **res)
    return {"status": st, "bits": bits, "enabled": bd.bd_debug_bounds_enabled(), "library": bd.LIB_PATH,
            "arrays": len(res)}


if __name__ == "__main__":
    print(json.dumps(run(sys.argv[1])))
