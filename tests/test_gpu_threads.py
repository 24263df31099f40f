"""Calls from several host threads at once, each thread on its own CUDA stream
with its own buffers (the header allows calls on distinct streams to run
concurrently): every result must equal what the same call gives alone, the
launch counter must count every launch, and the device error word stays 0.
Each thread also runs a decode-sized call of a different size, so that the
threads launch one kernel with different amounts of dynamic shared memory at
once.  The fused decode launch is not run concurrently (it is a cooperative
launch; nothing here depends on how two of them would share the SMs)."""
import threading

import pytest
import torch

from moe_routing_precision_gb300 import ops, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
THREADS = 4
ITERS = 6
T, E, K, H, N = 3000, 256, 8, 2048, 1024


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_routing_precision_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    assert ops.device_status() == 0
    yield
    assert ops.device_status() == 0


def _inputs(seed):
    inp = workloads.random_small(T, E, K, H, seed=seed, ties=seed % 2 == 1)
    g = torch.Generator().manual_seed(seed)
    y = torch.randn(T * K, H, generator=g).to(torch.bfloat16)
    xs = (torch.randn(T, 2 * N, generator=g) * 2).to(torch.bfloat16)
    return [t.to(DEV) for t in (inp["scores"], inp["x"], y, xs)]


def _chain(scores, x, y, xs, t_dec):
    """Every op once on the current stream; returns all outputs.  t_dec: the
    token count of a decode-sized call (a different one per thread, so the
    threads' launches need different amounts of shared memory)."""
    idx, w = ops.topk_gate(scores, K)
    counts, offsets, pos, src = ops.route_map(idx, E)
    q, sf = ops.expand_cast_fp8(x, pos)
    out = ops.combine(y, w, pos, torch.float32)
    q2, sf2 = ops.swiglu_cast_fp8(xs)
    q4, sf4 = ops.expand_cast_fp4(x, pos, group=32)
    dec = ops.route_expand_cast_fp8(scores[:t_dec].contiguous(), x[:t_dec].contiguous(), K)
    return [idx, w, counts, offsets, pos, src, q, sf, out, q2, sf2, q4, sf4, *dec]


def _same(a, b):
    return a.shape == b.shape and torch.equal(a.contiguous().view(torch.uint8),
                                              b.contiguous().view(torch.uint8))


def test_threads_on_distinct_streams_match_serial_results():
    inputs = [_inputs(100 + i) for i in range(THREADS)]
    t_dec = [100 + 300 * i for i in range(THREADS)]   # 100, 400, 700, 1000 tokens
    n0 = ops.launch_count()
    ref = [[t.clone() for t in _chain(*inp, td)] for inp, td in zip(inputs, t_dec)]
    torch.cuda.synchronize()
    total = ops.launch_count() - n0   # every thread's chain makes the same launches
    assert total > 0 and total % THREADS == 0
    per_chain = total // THREADS

    errors = []
    start = threading.Barrier(THREADS)

    def worker(i):
        try:
            torch.cuda.set_device(0)
            stream = torch.cuda.Stream(device=DEV)
            start.wait()
            with torch.cuda.stream(stream):
                for it in range(ITERS):
                    got = _chain(*inputs[i], t_dec[i])
                    stream.synchronize()
                    for j, (a, b) in enumerate(zip(got, ref[i])):
                        if not _same(a, b):
                            errors.append(f"thread {i} iteration {it} output {j} differs")
                            return
        except Exception as e:  # reported by the main thread
            errors.append(f"thread {i}: {type(e).__name__}: {e}")

    n1 = ops.launch_count()
    threads = [threading.Thread(target=worker, args=(i,)) for i in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads), "a worker thread did not finish"
    assert not errors, errors
    assert ops.launch_count() - n1 == per_chain * THREADS * ITERS
    assert ops.device_status() == 0
