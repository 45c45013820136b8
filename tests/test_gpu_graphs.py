"""The entry points inside a CUDA graph: once each shape has run once
(per-device facts and occupancies are cached on the first call), a captured
sequence of calls replays with new inputs written in place, and gives the
bits the same calls give when launched directly -- no host synchronisation,
allocation or query happens inside a call."""
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


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def inputs(seed, rows=96, H=512):
    x = synth.normal_with_outliers_bf16(seed, rows * H, 0.01, 50.0).reshape(rows, H)
    r = synth.normal_bf16(seed, 5, rows * H).reshape(rows, H)
    return x, r


def run_all(x, r, w, cos, sin, sc, sh, heads, D, S):
    """One call of every device entry point family on the current stream."""
    return [
        L.rms_norm(x, w, 1e-6),
        L.rms_norm_rope(x, w, cos, sin, heads, D, L.ROPE_INTERLEAVED, 1e-6, seq_len=S),
        L.rms_norm_rope(x, w, cos, sin, heads, D, L.ROPE_SPLIT_HALF, 1e-6, seq_len=S),
        L.rms_norm_adaln(x, None, sc, sh, 1e-6),
        L.add_rms_norm(x, r, w, 1e-6)[0],
        L.rope(x, heads, D, L.ROPE_SPLIT_HALF, (2, 6, 4), (10, 11, 11)),
        L.gelu_tanh(x),
    ]


def test_captured_calls_replay_with_new_inputs():
    heads, D, S = 8, 64, 48
    H = heads * D
    w = dev(synth.normal_bf16(401, 2, H, 1.0, 0.1))
    cos, sin = (torch.from_numpy(t).cuda() for t in synth.rope_table_1d(S, D))
    sc = dev(synth.normal_bf16(401, 3, 2 * H, 0.0, 0.5).reshape(2, H))
    sh = dev(synth.normal_bf16(401, 4, 2 * H, 0.0, 0.5).reshape(2, H))
    x0, r0 = inputs(402)
    x, r = dev(x0), dev(r0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run_all(x, r, w, cos, sin, sc, sh, heads, D, S)        # first calls: caches filled
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = run_all(x, r, w, cos, sin, sc, sh, heads, D, S)
    for seed in (403, 404):
        xn, rn = inputs(seed)
        x.copy_(dev(xn))
        r.copy_(dev(rn))
        g.replay()
        torch.cuda.synchronize()
        replayed = [bits(o) for o in outs]
        direct = [bits(o) for o in run_all(x, r, w, cos, sin, sc, sh, heads, D, S)]
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(replayed, direct)):
            assert np.array_equal(a, b), f"call {i}, inputs {seed}"
        # and the replayed norm is the oracle's
        assert compare_bf16(replayed[0], oracle.rms_norm(xn, bits(w), 1e-6))["ok"]


def test_concurrent_host_threads_on_separate_streams():
    """Calls from several host threads at once, each on its own stream:
    the per-device caches are shared under a lock and the last CUDA error is
    per thread, so every thread gets the results of a lone caller."""
    import threading
    heads, D, S = 8, 64, 48
    H = heads * D
    w = dev(synth.normal_bf16(411, 2, H, 1.0, 0.1))
    cos, sin = (torch.from_numpy(t).cuda() for t in synth.rope_table_1d(S, D))
    sc = dev(synth.normal_bf16(411, 3, 2 * H, 0.0, 0.5).reshape(2, H))
    sh = dev(synth.normal_bf16(411, 4, 2 * H, 0.0, 0.5).reshape(2, H))
    data = [tuple(dev(a) for a in inputs(420 + i)) for i in range(4)]
    expect = []
    for x, r in data:                      # one at a time
        expect.append([bits(o) for o in run_all(x, r, w, cos, sin, sc, sh, heads, D, S)])
    torch.cuda.synchronize()
    got, errors = [None] * len(data), []

    def work(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                x, r = data[i]
                for _ in range(20):
                    outs = run_all(x, r, w, cos, sin, sc, sh, heads, D, S)
                s.synchronize()
                got[i] = [bits(o) for o in outs]
        except Exception as e:             # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(data))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(len(data)):
        for a, b in zip(got[i], expect[i]):
            assert np.array_equal(a, b), f"thread {i}"
