"""Every entry point on page-locked host buffers: on GB300 the GPU addresses
pinned host memory directly (over NVLink-C2C), so a call given host x and y
streams them across the host link itself -- the way the bench's end-to-end
figures are taken.  The results must be the ones the same calls give on
device buffers, and the oracle's."""
import numpy as np
import pytest
import torch

import oracle
import rope_element_dit_gb300 as L
import synth
from oracle.compare import compare_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def pinned(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).pin_memory()


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def host_bits(t):
    return t.cpu().numpy().view(np.uint16)


def stream():
    return torch.cuda.current_stream().cuda_stream


def test_every_entry_point_on_pinned_host_buffers():
    rows, heads, D, S = 257, 16, 64, 64
    H = heads * D
    x = synth.normal_with_outliers_bf16(501, rows * H, 0.01, 50.0).reshape(rows, H)
    r = synth.normal_bf16(501, 5, rows * H).reshape(rows, H)
    w = synth.normal_bf16(501, 2, H, 1.0, 0.1)
    sc = synth.normal_bf16(501, 3, H, 0.0, 0.5).reshape(1, H)
    sh = synth.normal_bf16(501, 4, H, 0.0, 0.5).reshape(1, H)
    cos, sin = synth.rope_table_1d(S, D)
    hx, hr = pinned(x), pinned(r)
    wd, scd, shd = dev(w), dev(sc), dev(sh)
    cd, sd = torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda()
    out = {k: torch.empty(rows * H, dtype=torch.int16).pin_memory() for k in
           ("norm", "rope0", "rope1", "adaln", "add", "h", "pos", "gelu")}
    g_out = torch.empty(rows * H // 2, dtype=torch.int16).pin_memory()
    p = lambda t: t.data_ptr()
    calls = [
        L.ltxk_rms_norm(p(out["norm"]), p(hx), p(wd), rows, H, 1e-6, stream()),
        L.ltxk_rms_norm_rope_seq(p(out["rope0"]), p(hx), p(wd), p(cd), p(sd), rows, heads, D,
                                 0, 1e-6, S, stream()),
        L.ltxk_rms_norm_rope_seq(p(out["rope1"]), p(hx), p(wd), p(cd), p(sd), rows, heads, D,
                                 1, 1e-6, S, stream()),
        L.ltxk_rms_norm_adaln(p(out["adaln"]), p(hx), None, p(scd), p(shd), rows, H, rows,
                              1e-6, stream()),
        L.ltxk_add_rms_norm(p(out["add"]), p(out["h"]), p(hx), p(hr), p(wd), rows, H, 1e-6,
                            stream()),
        L.ltxk_rope(p(out["pos"]), p(hx), rows, heads, D, 1, 4, 4, 4, 10, 11, 11, 10000.0,
                    L.DTYPE_BF16, stream()),
        L.ltxk_gelu_tanh(p(out["gelu"]), p(hx), rows * H, stream()),
        L.ltxk_geglu(p(g_out), p(hx), rows, H // 2, stream()),
    ]
    assert all(st == L.OK for st in calls), [L.ltxk_status_string(st) for st in calls]
    torch.cuda.synchronize()
    got = {k: host_bits(v).reshape(rows, H) for k, v in out.items()}
    checks = {
        "norm": oracle.rms_norm(x, w, 1e-6),
        "rope0": oracle.rms_norm_rope(x, w, cos, sin, heads, D, 0, 1e-6),
        "rope1": oracle.rms_norm_rope(x, w, cos, sin, heads, D, 1, 1e-6),
        "gelu": oracle.gelu_tanh(x),
    }
    for k, ref in checks.items():
        assert compare_bf16(got[k], ref)["ok"], k
    y_ref, h_ref = oracle.add_rms_norm(x, r, w, 1e-6)
    assert np.array_equal(got["h"], h_ref) and compare_bf16(got["add"], y_ref)["ok"]
    assert compare_bf16(host_bits(g_out), oracle.geglu(x))["ok"]
    # AdaLN and the positional RoPE: the same bits as the calls on device buffers
    xd = dev(x)
    for k, call in (("adaln", lambda o: L.ltxk_rms_norm_adaln(o, xd.data_ptr(), None, p(scd),
                                                               p(shd), rows, H, rows, 1e-6,
                                                               stream())),
                    ("pos", lambda o: L.ltxk_rope(o, xd.data_ptr(), rows, heads, D, 1, 4, 4, 4,
                                                  10, 11, 11, 10000.0, L.DTYPE_BF16,
                                                  stream()))):
        od = torch.empty(rows * H, dtype=torch.int16, device="cuda")
        assert call(od.data_ptr()) == L.OK
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(od).reshape(rows, H), got[k]), k
