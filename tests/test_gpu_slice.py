"""GPU parity on the 70B-shaped decoder layer of the 8-layer slice workload:
the seven linears (q/o 8192x8192, k/v 1024x8192, gate/up 28672x8192, down
8192x28672), 14 variants compressed on the GPU from on-device seeded draws,
and 32 decode tokens spread over the variants by Zipf(1.1) with some
base-model tokens.  Compression is checked bit for bit (alpha to 1e-6) and the
multi-variant linear within the tolerances of tests/helpers.py, both on
sampled rows that always include the first and last row of each matrix.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_weight_delta_bd_gb300 import bitdelta as bd
from bit_weight_delta_bd_gb300 import synth
from helpers import check_linear, to_dev, u32, y_host

pytestmark = pytest.mark.gpu

V, T, SEED = 14, 32, 5


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("m", range(len(synth.SLICE_LINEARS)))
def test_slice_layer_linear(dev, m):
    name, d_out, d_in = synth.SLICE_LINEARS[m]
    scales = synth.slice_variant_scales(SEED, V)
    rows = synth.sample_rows(m, d_out, 24)
    wb = synth.device_base_weight(synth.slice_seed(SEED, 0, m), d_out, d_in, dev)
    wb_rows = _bits(wb[torch.from_numpy(rows).to(dev)])
    ws = bd.new_workspace(max(bd.bd_compress_workspace_size(d_out, d_in, bd.BD_ALPHA_PER_ROW),
                              bd.bd_linear_multi_workspace_size(T, V, d_out, d_in)), dev)
    signs, alphas, s_ref, a_ref = [], [], [], []
    for v in range(V):
        wf = synth.device_finetuned_weight(synth.slice_seed(SEED, 0, m, v), wb, float(scales[v]))
        s = torch.empty((d_out, d_in // 32), dtype=torch.int32, device=dev)
        a = torch.empty(d_out, dtype=torch.float32, device=dev)
        bd.bd_compress(wb, wf, bd.BD_ALPHA_PER_ROW, s, a, ws)
        wf_rows = _bits(wf[torch.from_numpy(rows).to(dev)])
        del wf
        sr, ar = oracle.compress_rows(wb_rows, wf_rows, np.arange(len(rows)))
        assert np.array_equal(u32(s)[rows], sr), f"{name} variant {v}: packed signs"
        np.testing.assert_allclose(a.cpu().numpy()[rows], ar, rtol=1e-6, atol=0)
        signs.append(s)
        alphas.append(a)
        sf = np.zeros((len(rows), d_in // 32), np.uint32)
        sf[:] = sr
        s_ref.append(sf)
        a_ref.append(ar)
    assert bd.bd_check_async(ws) == bd.BD_OK
    rng = np.random.default_rng(100 + m)
    vid = synth.zipf_variant_ids(rng, T, V)
    vid[[3, 17]] = -1  # two base-model tokens
    x = synth.activations(rng, T, d_in)
    y = torch.empty((T, d_out), dtype=torch.bfloat16, device=dev)
    bd.bd_linear_multi(to_dev(x, dev), to_dev(vid, dev), signs, alphas, bd.BD_ALPHA_PER_ROW, wb, y, ws)
    assert bd.bd_check_async(ws) == bd.BD_OK
    # oracle on the sampled rows only: a local W_base / signs / alpha of those rows
    y_ref = oracle.linear_multi(x, vid, s_ref, a_ref, True, wb_rows)
    check_linear(y_host(y)[:, rows], y_ref, bf16_out=True, what=f"slice {name}")
