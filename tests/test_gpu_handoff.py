"""The hand-off diagnostics (fm_test_pdl_chain, fm_test_grid_barrier).

CPU: argument checks return their status without touching a GPU. GPU: every CTA of a
cooperative launch completes every barrier round in both orderings; a CTA that never
arrives makes every bounded wait run out (FM_ERR_DEVICE, promptly, and the context
stays usable: the next launch succeeds); the dependent-launch chain times positive."""
import ctypes

import numpy as np
import pytest

import flow_matching_action_denoise_gb300 as fmad


def test_host_argument_checks():
    L = fmad.load()
    us = ctypes.c_float()
    assert L.fm_test_pdl_chain(1, 32, 0, 1, 1, 1, 0, 16, 4, ctypes.byref(us)) == 2     # FM_ERR_SHAPE
    assert L.fm_test_pdl_chain(1, 32, 1, 1, 1, 1, 0, None, 4, ctypes.byref(us)) == 1   # FM_ERR_INVALID_ARG
    assert L.fm_test_pdl_chain(1, 48, 1, 1, 1, 1, 0, 16, 4, ctypes.byref(us)) == 2     # threads not a multiple of 32
    assert L.fm_test_pdl_chain(6, 32, 1, 1, 1, 4, 0, 16, 4, ctypes.byref(us)) == 2     # cluster does not divide ctas
    assert L.fm_test_pdl_chain(8, 32, 1, 1, 1, 8, 2, 16, 64, ctypes.byref(us)) == 4    # FM_ERR_WORKSPACE
    assert L.fm_test_grid_barrier(1, 32, 1, 0, 10 ** 6, None, 16, None) == 1
    assert L.fm_test_grid_barrier(1, 32, 1, 3, 10 ** 6, 16, 16, None) == 2          # mode
    assert L.fm_test_grid_barrier(1, 32, 1, 0, 10, 16, 16, None) == 2               # budget below 1 us
    assert L.fm_test_grid_barrier(1, 32, 1, 0, 10 ** 6, 8, 16, None) == 3           # scratch alignment


def _bufs(ctas):
    import torch
    scratch = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.zeros(2 * ctas, dtype=torch.int64, device="cuda")
    return scratch, out


@pytest.mark.gpu
@pytest.mark.parametrize("mode", [0, 1])
def test_grid_barrier_completes_every_round(mode):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for ctas in (8, sms):
        scratch, out = _bufs(ctas)
        assert fmad.grid_barrier(ctas, 256, 200, mode, 10 ** 9, scratch, out) == 0
        o = out.cpu().numpy().reshape(ctas, 2)
        assert np.all(o[:, 1] == 200)
        assert np.all(o[:, 0] > 0)
        assert scratch.cpu().numpy()[0] == 200 * ctas   # every arrival counted once
        assert scratch.cpu().numpy()[1] == 0


@pytest.mark.gpu
def test_grid_barrier_wait_runs_out_and_context_survives():
    import time
    scratch, out = _bufs(16)
    t0 = time.perf_counter()
    assert fmad.grid_barrier(16, 128, 3, 2, 2 * 10 ** 6, scratch, out) == 7   # FM_ERR_DEVICE
    assert time.perf_counter() - t0 < 5.0
    o = out.cpu().numpy().reshape(16, 2)
    assert np.all(o[:, 1] == 0)                 # no CTA got past the first barrier
    assert scratch.cpu().numpy()[1] == 1        # the error word
    assert scratch.cpu().numpy()[0] == 15       # CTA 0 never arrived
    assert fmad.grid_barrier(16, 128, 5, 0, 10 ** 9, scratch, out) == 0
    assert np.all(out.cpu().numpy().reshape(16, 2)[:, 1] == 5)


@pytest.mark.gpu
def test_grid_barrier_rejects_more_ctas_than_fit():
    scratch, out = _bufs(1)
    with pytest.raises(fmad.FmError):
        fmad.grid_barrier(1 << 20, 1024, 1, 0, 10 ** 6, scratch, out)


@pytest.mark.gpu
@pytest.mark.parametrize("pdl,cluster,writes", [(True, 1, 0), (False, 1, 0), (True, 8, 4)])
def test_pdl_chain_times_positive(pdl, cluster, writes):
    import torch
    scratch = torch.zeros(1 + 64 * 128 * writes, dtype=torch.int32, device="cuda")
    us = fmad.pdl_chain(64, 128, 100, 3, pdl, scratch, cluster, writes)
    assert np.isfinite(us) and 0.0 < us < 1000.0
    assert int(scratch[0].item()) == 100 * 4    # the warm-up run and three timed runs
    if writes:
        w = scratch[1:].cpu().numpy().reshape(writes, 64 * 128)
        assert np.all(w == np.arange(writes)[:, None])
