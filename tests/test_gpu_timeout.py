"""The bounded-wait (timeout) path of the kernels, exercised without a fault.

tq_debug_stall_next_launch makes the next matmul kernel's first thread block
request none of its input copies, so its waits run out against a barrier
that nothing completes. The test checks that the launch still ends promptly
(the block gives up after the short limit and waits only for copies it did
request), that tq_device_status reports TQ_ERR_TIMEOUT once and then clears,
and that the next call on the same context gives the exact results again.
Nothing here faults, traps or waits without bound.
"""
import time

import numpy as np
import pytest

import synth

STALL_NS = 200_000   # 200 us


@pytest.fixture(scope="module")
def tq():
    from bit_matvec_gb300 import build
    build.build()
    import bit_matvec_gb300
    return bit_matvec_gb300


def test_stall_argument_checked(tq):
    with pytest.raises(tq.TQError):
        tq.tq_debug_stall_next_launch(-1)
    tq.tq_debug_stall_next_launch(0)   # cancels; no launch involved


# (rows, cols, ntok): the one-token dp4a GEMV, the mma.sync GEMV (staging its
# activations itself at 1024 columns; loading them from the workspace, where
# a staging kernel wrote them, at 5120), the tensor-core kernel of the
# workspace form (two token tiles)
CASES = [(4096, 8192, 1), (4096, 1024, 4), (4096, 5120, 4), (1024, 1024, 100)]


@pytest.mark.gpu
@pytest.mark.parametrize("rows,cols,ntok", CASES)
def test_timeout_reported_then_cleared(tq, rows, cols, ntok):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gpu_util import DEV, gpu_quantize, gpu_repack

    s = synth.seeds(2)
    wpq = synth.pq2_0_weights(rows, cols, 2)
    x = synth.activations(ntok, cols, s["acts"])
    Wtq, Xq = gpu_repack(wpq, rows, cols), gpu_quantize(x)
    ws = tq.workspace_empty(rows, cols, ntok, DEV)

    def run():
        Y = torch.full((ntok, rows), float("nan"), dtype=torch.float32, device=DEV)
        tq.tq_matmul_ws(Wtq, Xq, Y, rows, cols, ntok, ws)
        return Y

    y0 = run().cpu().numpy()
    assert tq.tq_device_status() == tq.TQ_OK

    torch.cuda.synchronize()
    tq.tq_debug_stall_next_launch(STALL_NS)
    try:
        t0 = time.perf_counter()
        run()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        tq.tq_debug_stall_next_launch(0)
    assert tq.tq_device_status() == tq.TQ_ERR_TIMEOUT
    # the stalled block gave up after 200 us and waited for nothing it had not
    # requested (the regular limit is 2 s)
    assert dt < 1.0, f"stalled launch took {dt:.3f} s"
    assert tq.tq_device_status() == tq.TQ_OK   # read and cleared

    y1 = run().cpu().numpy()
    assert tq.tq_device_status() == tq.TQ_OK
    assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))
