"""The allocation-free RMSNorm entry point, ltxk_rms_norm_noalloc.

It serves callers that cannot allocate device memory: engines whose device
memory all comes from their own pre-sized pool, and latency-critical loops
that cannot take an allocation's implicit synchronisation.  Its kernel's only
extra device memory is a fault word kept in the library's static device
array.  This file is collected last, so a run that stops at the first failure
has run every other test before it; it also passes on its own in a fresh
process (the first call on the device does the set-up).
"""
import numpy as np
import pytest
import torch

import rope_element_dit_gb300 as L
import synth
from oracle.compare import compare_bf16

pytestmark = pytest.mark.gpu


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


@pytest.mark.parametrize("rows,hidden,with_w", [(4099, 3072, True), (1000, 2048, False),
                                                (37, 264, True), (5, 4096, True)])
def test_noalloc_matches_rms_norm_on_two_calls(rows, hidden, with_w):
    assert torch.cuda.is_available()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        seed = 4200 + 10 * call + rows % 7
        x = _dev(synth.normal_bf16(seed, 0, rows * hidden).reshape(rows, hidden))
        w = _dev(synth.normal_bf16(seed, 2, hidden, 1.0, 0.1)) if with_w else None
        ref = torch.empty_like(x)
        got = torch.full_like(x, 0x7FC1)
        wp = None if w is None else w.data_ptr()
        assert L.ltxk_rms_norm(ref.data_ptr(), x.data_ptr(), wp, rows, hidden, 1e-6,
                               stream) == L.OK
        assert L.ltxk_rms_norm_noalloc(got.data_ptr(), x.data_ptr(), wp, rows, hidden,
                                       1e-6, stream) == L.OK
        torch.cuda.synchronize()
        r = compare_bf16(got.cpu().numpy().view(np.uint16), ref.cpu().numpy().view(np.uint16))
        assert r["ok"], f"call {call}: {r}"


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
