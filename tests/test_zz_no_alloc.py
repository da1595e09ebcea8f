"""bd_compress_noalloc: compression for callers that cannot allocate device
memory (an allocator owned by a framework, stream capture, a C host without
its own device allocator).  It keeps its partial sums in a fixed array of the
library instead of a caller workspace; these checks call it through the C ABI
twice in a row and compare every output with bd_compress and with the CPU
oracle, also at the largest row count the fixed array serves.

The file name makes pytest collect it last, so a run that stops at the first
failure has run every other test before this one.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_weight_delta_bd_gb300 import bitdelta as bd
from bit_weight_delta_bd_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _d(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)


@pytest.mark.parametrize("mode", [bd.BD_ALPHA_PER_MATRIX, bd.BD_ALPHA_PER_ROW])
def test_noalloc_matches_workspace_entry_point_twice(dev, mode):
    lib = bd.load()
    st = torch.cuda.current_stream().cuda_stream
    # two calls in a row, different shapes, so the second reuses the scratch left by the first
    for call, (d_out, d_in) in enumerate([(1000, 1024), (37, 384)]):
        wb, wf, _ = synth.single_problem(50 + call, d_out, d_in, 1)
        wb_d, wf_d = _d(wb, dev), _d(wf, dev)
        n_a = d_out if mode == bd.BD_ALPHA_PER_ROW else 1
        s_ref = torch.empty((d_out, d_in // 32), dtype=torch.int32, device=dev)
        a_ref = torch.empty(n_a, dtype=torch.float32, device=dev)
        ws = bd.new_workspace(bd.bd_compress_workspace_size(d_out, d_in, mode), dev)
        bd.bd_compress(wb_d, wf_d, mode, s_ref, a_ref, ws)
        assert bd.bd_check_async(ws) == bd.BD_OK
        s = torch.full((d_out, d_in // 32), 7, dtype=torch.int32, device=dev)
        a = torch.full((n_a,), -1.0, dtype=torch.float32, device=dev)
        assert lib.bd_compress_noalloc(wb_d.data_ptr(), wf_d.data_ptr(), d_out, d_in, mode, s.data_ptr(),
                                       a.data_ptr(), st) == bd.BD_OK
        torch.cuda.synchronize()
        assert torch.equal(s, s_ref), f"call {call}: packed signs differ"
        np.testing.assert_allclose(a.cpu().numpy(), a_ref.cpu().numpy(), rtol=1e-6, atol=0)
        so, ao = oracle.compress(wb, wf, per_row=mode == bd.BD_ALPHA_PER_ROW)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), so), f"call {call}: signs differ from the oracle"
        np.testing.assert_allclose(a.cpu().numpy(), ao, rtol=1e-6, atol=0)


@pytest.mark.parametrize("d_out", [bd.BD_NOALLOC_MAX_ROWS, bd.BD_NOALLOC_MAX_ROWS - 3])
def test_noalloc_at_the_row_limit_matches_the_oracle(dev, d_out):
    """Every partial sum of the fixed array in use (per-matrix alpha over the
    largest row count it serves, and a ragged count just below it), two calls
    in a row, against the oracle: bits exact, alpha to 1e-6 relative."""
    lib = bd.load()
    st = torch.cuda.current_stream().cuda_stream
    d_in = 128
    wb, wf, _ = synth.single_problem(d_out % 1000, d_out, d_in, 1)
    so, ao = oracle.compress(wb, wf, per_row=False)
    wb_d, wf_d = _d(wb, dev), _d(wf, dev)
    for call in range(2):
        s = torch.full((d_out, d_in // 32), 7, dtype=torch.int32, device=dev)
        a = torch.full((1,), -1.0, dtype=torch.float32, device=dev)
        assert lib.bd_compress_noalloc(wb_d.data_ptr(), wf_d.data_ptr(), d_out, d_in, bd.BD_ALPHA_PER_MATRIX,
                                       s.data_ptr(), a.data_ptr(), st) == bd.BD_OK
        torch.cuda.synchronize()
        assert np.array_equal(s.cpu().numpy().view(np.uint32), so), f"call {call}: packed signs"
        np.testing.assert_allclose(a.cpu().numpy(), ao, rtol=1e-6, atol=0)


def test_noalloc_rejects_more_rows_than_its_scratch(dev):
    lib = bd.load()
    st = torch.cuda.current_stream().cuda_stream
    big = bd.BD_NOALLOC_MAX_ROWS + 1
    # the size check comes before any pointer is touched
    assert lib.bd_compress_noalloc(1 << 40, 1 << 41, big, 128, bd.BD_ALPHA_PER_MATRIX, 1 << 42, 1 << 43, st) == \
        bd.BD_ERR_UNSUPPORTED_SHAPE
