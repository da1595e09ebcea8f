"""Delta cache policy on the CPU (bd_cache_* in dry-run mode: no arena, no
CUDA call).  The rules come from section "Altyapı ayrıntıları" of the
BitDelta post: a delta is loaded on its variant's first request and stays
until evicted; eviction is request-rate-weighted LRU with the most requested
variants pinned (the post keeps the top 6 of 14 resident); requests for a
variant whose delta is loading wait for that one load."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from bit_weight_delta_bd_gb300 import bitdelta as bd

SLOT = 1 << 20


def make_cache(n_slots, n_pinned, variants, decay=1.0):
    c = bd.DeltaCache(None, SLOT, n_pinned, decay, n_slots=n_slots)
    for v in variants:
        c.set_source(v, torch.zeros(1024, dtype=torch.uint8))
    return c


def step(c, vids):
    d, s = c.step(vids)
    c.release()
    return d, s


def resident(c, variants):
    return {v for v in variants if c.query(v)[0]}


def test_cold_start_then_hits():
    c = make_cache(4, 0, range(3))
    d, s = step(c, [1])
    assert list(s) == [bd.BD_CACHE_SERVED] and d[0] is not None
    st = c.stats()
    assert (st["loads"], st["misses"], st["hits"], st["bytes_loaded"]) == (1, 1, 0, 1024)
    d2, _ = step(c, [1, 1])
    assert d2 == [d[0], d[0]]
    st = c.stats()
    assert (st["loads"], st["hits"]) == (1, 2)


def test_one_load_for_many_requests_and_base_tokens():
    c = make_cache(4, 0, range(5))
    d, s = step(c, [3] * 10 + [-1, -1])
    assert list(s) == [bd.BD_CACHE_SERVED] * 10 + [bd.BD_CACHE_BASE] * 2
    assert len({x for x in d[:10]}) == 1 and d[10] is None
    st = c.stats()
    assert (st["loads"], st["misses"], st["requests"]) == (1, 10, 10)


def test_lru_evicts_the_least_recently_used():
    c = make_cache(3, 0, range(5))
    for v in (0, 1, 2, 0):
        step(c, [v])
    assert resident(c, range(5)) == {0, 1, 2}
    step(c, [3])  # 1 is the least recently used
    assert resident(c, range(5)) == {0, 2, 3}
    step(c, [4])  # then 2
    assert resident(c, range(5)) == {0, 3, 4}
    assert c.stats()["evictions"] == 2


def test_top_six_of_fourteen_stay_resident():
    """14 variants, 8 slots, 6 pinned: heavy traffic on variants 0-5, the
    other 8 requested one at a time in turn.  The heavy six stay resident and
    pinned; the two free slots hold the two most recently requested others."""
    c = make_cache(8, 6, range(14), decay=0.9)
    rng = np.random.default_rng(0)
    for k in range(60):
        light = 6 + k % 8
        vids = list(rng.integers(0, 6, size=24)) + [light]
        d, s = step(c, vids)
        assert all(x == bd.BD_CACHE_SERVED for x in s)
        if k >= 10:
            res = resident(c, range(14))
            assert set(range(6)) <= res
            assert all(c.query(v)[1] for v in range(6))
            assert res - set(range(6)) == {light, 6 + (k - 1) % 8}
    st = c.stats()
    assert st["pinned"] == 6 and st["resident"] == 8
    # the heavy six were loaded once each; every light request after the
    # first round was a miss
    assert st["loads"] == 6 + 60


def test_pinned_slots_are_not_evicted_requests_queue():
    c = make_cache(2, 2, range(4))
    for _ in range(3):
        step(c, [0, 0, 1])
    d, s = step(c, [2, 2, 0])
    assert list(s) == [bd.BD_CACHE_QUEUED, bd.BD_CACHE_QUEUED, bd.BD_CACHE_SERVED]
    assert d[0] is None and d[2] is not None
    assert resident(c, range(4)) == {0, 1}
    assert c.stats()["queued"] == 2


def test_more_variants_than_slots_most_requested_first():
    c = make_cache(2, 0, range(4))
    d, s = step(c, [3, 1, 1, 2, 1, 2])
    # 1 (3 requests) and 2 (2 requests) get the two slots, 3 waits
    assert list(s) == [bd.BD_CACHE_QUEUED] + [bd.BD_CACHE_SERVED] * 5
    assert resident(c, range(4)) == {1, 2}


def test_pinned_set_follows_the_request_rate():
    c = make_cache(3, 1, range(3), decay=0.5)
    for _ in range(4):
        step(c, [0, 0, 0, 1])
    assert c.query(0)[1] and not c.query(1)[1]
    for _ in range(4):
        step(c, [1, 1, 1, 0])
    assert c.query(1)[1] and not c.query(0)[1]


def test_step_needs_release_and_rejects_bad_ids():
    c = make_cache(2, 0, range(2))
    c.step([0])
    with pytest.raises(bd.BitDeltaError):
        c.step([1])
    c.release()
    c.step([1])
    c.release()
    before = c.stats()
    with pytest.raises(bd.BitDeltaError):
        c.step([5])  # no source registered
    with pytest.raises(bd.BitDeltaError):
        c.step([-2])
    assert c.stats() == before  # a rejected step changes nothing


def test_failed_load_hands_out_nothing_and_needs_no_release():
    """A copy that fails (a host-side fake of the failing call) ends the
    step with BD_ERR_CUDA: nothing is handed out, so the next step runs
    without a release; the load issued before the failure stays resident,
    the slot whose load failed is empty, later variants were not loaded."""
    c = make_cache(4, 0, range(8))
    step(c, [0, 1])
    c.debug_fail_load(2)
    with pytest.raises(bd.BitDeltaError) as ei:
        c.step([2, 2, 3, 4])  # 2 loads, 3 fails, 4 is never reached
    assert ei.value.status == bd.BD_ERR_CUDA
    assert resident(c, range(8)) == {0, 1, 2}
    st = c.stats()
    assert st["loads"] == 3 and st["resident"] == 3
    d, s = step(c, [3, 0])  # no release needed; the empty slot takes 3
    assert list(s) == [bd.BD_CACHE_SERVED, bd.BD_CACHE_SERVED]
    assert resident(c, range(8)) == {0, 1, 2, 3}
    assert c.stats()["loads"] == 4


def test_create_and_source_errors():
    with pytest.raises(bd.BitDeltaError):
        bd.DeltaCache(None, 0, 0, n_slots=4)
    with pytest.raises(bd.BitDeltaError):
        bd.DeltaCache(None, SLOT, 0, rate_decay=1.5, n_slots=4)
    c = make_cache(2, 0, [0])
    with pytest.raises(bd.BitDeltaError):
        c.set_source(1, torch.zeros(SLOT + 1, dtype=torch.uint8))  # larger than a slot
    step(c, [0])
    with pytest.raises(bd.BitDeltaError):
        c.set_source(0, torch.zeros(16, dtype=torch.uint8))  # resident


def _dyadic_variants(seed, V, d_out, d_in):
    """W_base in {k/64 : |k| <= 8} and W_v = W_base +- 2^-(3 + v mod 6): with
    integer activations every partial sum of the fused linear is exact in
    fp32, so the GPU result must equal the fp64 oracle bit for bit."""
    from bit_weight_delta_bd_gb300 import synth

    rng = np.random.default_rng(seed)
    wb = rng.integers(-8, 9, size=(d_out, d_in)).astype(np.float32) / 64.0
    wfs = []
    for v in range(V):
        s = np.where(rng.random((d_out, d_in)) < 0.5, -1.0, 1.0).astype(np.float32)
        wfs.append(synth.f32_to_bf16_bits(wb + s * 2.0 ** -(3 + v % 6)))
    return synth.f32_to_bf16_bits(wb), wfs


@pytest.mark.gpu
def test_cache_serves_bd_linear_multi_bit_identical():
    """Real arena (8 slots, 6 pinned) in front of bd_linear_multi: 14
    variants' packed signs and alphas live in pinned host memory and are
    loaded on demand on a copy stream.  Every step's output equals the fp64
    oracle on the same tokens bit for bit (exact dyadic inputs) and the same
    call on device-resident deltas; queued requests are served by a later
    step."""
    import ctypes

    import oracle
    from bit_weight_delta_bd_gb300 import synth

    assert torch.cuda.is_available()
    import __graft_entry__

    __graft_entry__.build()
    dev = torch.device("cuda:0")
    V, d_out, d_in, T = 14, 512, 1024, 32
    wb, wfs = _dyadic_variants(5, V, d_out, d_in)
    refs = [oracle.compress(wb, wf, per_row=True) for wf in wfs]
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)  # noqa: E731
    wb_d = to(wb)
    ws = bd.new_workspace(max(bd.bd_compress_workspace_size(d_out, d_in, bd.BD_ALPHA_PER_ROW),
                              bd.bd_linear_multi_workspace_size(T, V, d_out, d_in)), dev)
    signs = [torch.empty((d_out, d_in // 32), dtype=torch.int32, device=dev) for _ in range(V)]
    alphas = [torch.empty(d_out, dtype=torch.float32, device=dev) for _ in range(V)]
    for v in range(V):
        bd.bd_compress(wb_d, to(wfs[v]), bd.BD_ALPHA_PER_ROW, signs[v], alphas[v], ws)
    assert bd.bd_check_async(ws) == bd.BD_OK
    for v in range(V):
        assert np.array_equal(signs[v].cpu().numpy().view(np.uint32), refs[v][0])
        assert np.array_equal(alphas[v].cpu().numpy(), refs[v][1])
    sbytes = d_out * d_in // 8
    slot = (sbytes + 4 * d_out + 255) // 256 * 256
    blobs = []
    for v in range(V):
        h = torch.empty(sbytes + 4 * d_out, dtype=torch.uint8, pin_memory=True)
        h[:sbytes] = signs[v].view(torch.uint8).reshape(-1).cpu()
        h[sbytes:] = alphas[v].view(torch.uint8).cpu()
        blobs.append(h)
    arena = torch.zeros(8 * slot, dtype=torch.uint8, device=dev)
    copy_stream = torch.cuda.Stream()
    cache = bd.DeltaCache(arena, slot, 6, 0.9, copy_stream=copy_stream)
    for v in range(V):
        cache.set_source(v, blobs[v])
    lib = bd.load()
    rng = np.random.default_rng(9)
    pending = []  # (vid, x) of queued requests
    served_total = 0
    for k in range(30):
        new_vid = synth.zipf_variant_ids(rng, T, V)
        new_vid[rng.random(T) < 0.1] = -1
        new_x = synth.f32_to_bf16_bits(rng.integers(-4, 5, size=(T, d_in)).astype(np.float32))
        vids = np.concatenate([np.array([p[0] for p in pending], np.int32), new_vid]) if pending else new_vid
        xs = np.concatenate([np.stack([p[1] for p in pending]), new_x]) if pending else new_x
        ptr, state = cache.step(vids)
        ok = state != bd.BD_CACHE_QUEUED
        pending = [(int(vids[i]), xs[i]) for i in range(len(vids)) if not ok[i]]
        sv, sx = vids[ok], xs[ok]
        served_total += len(sv)
        base = next((p for p in ptr if p is not None), arena.data_ptr())
        s_tab = (ctypes.c_void_p * V)(*[base] * V)
        a_tab = (ctypes.c_void_p * V)(*[base + sbytes] * V)
        for i in range(len(vids)):
            if ok[i] and vids[i] >= 0:
                s_tab[vids[i]] = ptr[i]
                a_tab[vids[i]] = ptr[i] + sbytes
        x_d, v_d = to(sx), torch.from_numpy(sv).to(dev)
        y = torch.empty((len(sv), d_out), dtype=torch.float32, device=dev)
        st = torch.cuda.current_stream().cuda_stream
        assert lib.bd_linear_multi(x_d.data_ptr(), len(sv), v_d.data_ptr(), V, ctypes.addressof(s_tab),
                                   ctypes.addressof(a_tab), bd.BD_ALPHA_PER_ROW, wb_d.data_ptr(), d_out, d_in,
                                   y.data_ptr(), bd.BD_OUT_F32, ws.data_ptr(), ws.numel(), st) == bd.BD_OK
        cache.release()
        y_ref = torch.empty_like(y)
        bd.bd_linear_multi(x_d, v_d, signs, alphas, bd.BD_ALPHA_PER_ROW, wb_d, y_ref, ws)
        assert bd.bd_check_async(ws) == bd.BD_OK
        y_host = y.cpu().numpy().astype(np.float64)
        y_oracle = oracle.linear_multi(sx, sv, [r[0] for r in refs], [r[1] for r in refs], True, wb)
        assert np.array_equal(y_host, y_oracle), f"step {k}: differs from the oracle"
        assert torch.equal(y, y_ref), f"step {k}: differs from the resident-delta call"
    st = cache.stats()
    assert st["pinned"] == 6 and st["resident"] <= 8 and st["loads"] >= 6
    assert served_total + len(pending) == 30 * T
    cache.close()
