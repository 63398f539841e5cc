"""Concurrent use of the library from several host threads and streams.

The library keeps per-device caches (kernel attributes, occupancy, the device
check) that the first call on a device fills; ctypes releases the interpreter
lock during the call, so threads really do enter the library at once. Each
thread runs the MLP on its own stream with its own workspace and output; every
result must equal the one computed alone, bit for bit.
"""

import threading

import pytest

import synth
from mxutil import bf16_to_device

pytestmark = pytest.mark.gpu


def test_threads_on_separate_streams_match_serial(lib):
    import torch

    n_threads, M, d, ff = 4, 512, 512, 1024
    w = synth.full_mlp(M=M, d=d, ff=ff)
    w1 = lib.mx_quantize(bf16_to_device(w["w1"]))
    w2 = lib.mx_quantize(bf16_to_device(w["w2"]))
    b1, b2 = bf16_to_device(w["b1"]), bf16_to_device(w["b2"])
    xs = [bf16_to_device(synth.full_mlp(seed=10 + i, M=M, d=d, ff=ff)["x"]) for i in range(n_threads)]
    need = lib.mx_mlp_workspace_bytes(M, d, ff)
    torch.cuda.synchronize()

    ref = []
    for x in xs:
        ref.append(lib.mx_mlp(x, w1, b1, w2, b2))
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream() for _ in range(n_threads)]
    outs = [torch.empty_like(x) for x in xs]
    wss = [torch.empty(need, dtype=torch.uint8, device="cuda") for _ in range(n_threads)]
    errors = []
    start = threading.Barrier(n_threads)

    def worker(i):
        try:
            torch.cuda.set_device(0)
            start.wait()
            for _ in range(5):
                lib.mx_mlp(xs[i], w1, b1, w2, b2, y=outs[i], workspace=wss[i], stream=streams[i])
            streams[i].synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(n_threads)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    assert all(not t.is_alive() for t in threads)
    torch.cuda.synchronize()
    for i in range(n_threads):
        assert torch.equal(outs[i], ref[i]), f"thread {i} differs from the serial result"
    assert lib.mx_device_error() == 0
