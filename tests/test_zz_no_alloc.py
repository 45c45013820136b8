"""The allocation-free RMSNorm entry point, ltxk_rms_norm_noalloc.

It serves callers that cannot allocate device memory: engines whose device
memory all comes from their own pre-sized pool, and latency-critical loops
that cannot take an allocation's implicit synchronisation.  Its kernel's only
extra device memory is a fault word kept in the library's static device
array, which ltxk_noalloc_fault_status reads back.  This file is collected
last, so a run that stops at the first failure has run every other test
before it; it also passes on its own in a fresh process (the first call on
the device does the set-up).
"""
import numpy as np
import pytest
import torch

import oracle
import rope_element_dit_gb300 as L
import synth
from oracle.compare import compare_bf16

pytestmark = pytest.mark.gpu


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _host(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("rows,hidden,with_w", [(4099, 3072, True), (1000, 2048, False),
                                                (37, 264, True), (5, 4096, True)])
def test_noalloc_matches_the_oracle_and_rms_norm_on_two_calls(rows, hidden, with_w):
    assert torch.cuda.is_available()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        seed = 4200 + 10 * call + rows % 7
        xb = synth.normal_bf16(seed, 0, rows * hidden).reshape(rows, hidden)
        wb = synth.normal_bf16(seed, 2, hidden, 1.0, 0.1) if with_w else None
        x = _dev(xb)
        w = None if wb is None else _dev(wb)
        ref = torch.empty_like(x)
        got = torch.full_like(x, 0x7FC1)
        wp = None if w is None else w.data_ptr()
        assert L.ltxk_rms_norm(ref.data_ptr(), x.data_ptr(), wp, rows, hidden, 1e-6,
                               stream) == L.OK
        assert L.ltxk_rms_norm_noalloc(got.data_ptr(), x.data_ptr(), wp, rows, hidden,
                                       1e-6, stream) == L.OK
        assert L.ltxk_noalloc_fault_status() == L.OK
        torch.cuda.synchronize()
        want = oracle.rms_norm(xb, wb, 1e-6)
        r = compare_bf16(_host(got), want)
        assert r["ok"], f"call {call} vs the oracle: {r}"
        r = compare_bf16(_host(got), _host(ref))
        assert r["ok"], f"call {call} vs ltxk_rms_norm: {r}"


def test_noalloc_in_place_over_several_passes_of_the_ring():
    # 4099 rows of 3072: more rows than one pass of the persistent grid, so
    # the ring refills its buffers from x while earlier rows are written
    rows, hidden = 4099, 3072
    xb = synth.normal_bf16(4300, 0, rows * hidden).reshape(rows, hidden)
    wb = synth.normal_bf16(4300, 2, hidden, 1.0, 0.1)
    x = _dev(xb)
    w = _dev(wb)
    s = torch.cuda.current_stream().cuda_stream
    assert L.ltxk_rms_norm_noalloc(x.data_ptr(), x.data_ptr(), w.data_ptr(), rows, hidden,
                                   1e-6, s) == L.OK
    assert L.ltxk_noalloc_fault_status() == L.OK
    r = compare_bf16(_host(x), oracle.rms_norm(xb, wb, 1e-6))
    assert r["ok"], r


def test_noalloc_wait_that_runs_out_is_reported_and_cleared():
    # The diagnostic leaves every warp's first bulk copy unissued: those
    # waits run out after 50 ms, the kernel returns, and the fault word in
    # the static array says so -- once.
    rows, hidden = 4 * 152 * 2 * 8, 1024      # several rows per warp
    xb = synth.normal_bf16(4400, 0, rows * hidden).reshape(rows, hidden)
    x = _dev(xb)
    y = torch.zeros_like(x)
    s = torch.cuda.current_stream().cuda_stream
    assert L.ltxk_noalloc_fault_status() == L.OK
    assert L.ltxk_diag_noalloc_missing_copy(y.data_ptr(), x.data_ptr(), rows, hidden,
                                            50_000_000, s) == L.OK
    assert L.ltxk_noalloc_fault_status() == L.ERR_TIMEOUT
    assert L.ltxk_noalloc_fault_status() == L.OK
    # the context still works, and the next call starts from a clear word
    assert L.ltxk_rms_norm_noalloc(y.data_ptr(), x.data_ptr(), None, rows, hidden, 1e-6,
                                   s) == L.OK
    assert L.ltxk_noalloc_fault_status() == L.OK
    r = compare_bf16(_host(y), oracle.rms_norm(xb, None, 1e-6))
    assert r["ok"], r


def test_noalloc_rejects_what_it_does_not_handle():
    x = torch.zeros(8 * 4104, dtype=torch.int16, device="cuda")
    y = torch.zeros_like(x)
    s = torch.cuda.current_stream().cuda_stream
    # rows wider than the maximum, or not whole 16-byte vectors
    assert L.ltxk_rms_norm_noalloc(y.data_ptr(), x.data_ptr(), None, 8, 4104, 1e-6,
                                   s) == L.ERR_SHAPE
    assert L.ltxk_rms_norm_noalloc(y.data_ptr(), x.data_ptr(), None, 8, 12, 1e-6,
                                   s) == L.ERR_SHAPE
    # pointers off a 16-byte boundary
    assert L.ltxk_rms_norm_noalloc(y.data_ptr() + 2, x.data_ptr(), None, 4, 8, 1e-6,
                                   s) == L.ERR_ALIGN
    assert L.ltxk_rms_norm_noalloc(y.data_ptr(), x.data_ptr(), None, 0, 8, 1e-6, s) == L.OK
    # the diagnostic's wait limit must be in range
    assert L.ltxk_diag_noalloc_missing_copy(y.data_ptr(), x.data_ptr(), 4, 8, 10,
                                            s) == L.ERR_SHAPE
