"""tq_matmul_static_ws: the matmul whose workspace is the library's own fixed
device array, for callers that cannot allocate device memory.

On the GPU it must give what tq_matmul_ws gives with a caller workspace, on
consecutive calls that reuse the shared array with different shapes (the
second call finds the first one's contents there). Host side: sizes beyond
the array are rejected before any CUDA work. This file runs last so that the
array is first used after the other tests, and also passes on its own.
"""
import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tq():
    from bit_matvec_gb300 import build
    build.build()
    import bit_matvec_gb300
    return bit_matvec_gb300


def test_limit_matches_header(tq):
    with open(os.path.join(ROOT, "include", "tq.h")) as f:
        m = re.search(r"#define\s+TQ_STATIC_WS_BYTES\s+\((\d+)\s*<<\s*(\d+)\)", f.read())
    assert m and int(m.group(1)) << int(m.group(2)) == tq.STATIC_WS_BYTES


def test_oversize_rejected_before_any_cuda_work(tq):
    """Rejected shapes return before the array is looked up or anything is
    launched, so NULL pointers are safe here."""
    lib = tq.library()
    assert tq.tq_matmul_workspace_bytes(64, 5120, 768) <= tq.STATIC_WS_BYTES
    assert tq.tq_matmul_workspace_bytes(64, 5120, 769) > tq.STATIC_WS_BYTES
    for rows, cols, ntok in [(64, 5120, 769), (1, 256 * 1024, 17), (1, 256, 1 << 40),
                             (1, 1 << 40, 1 << 40)]:
        assert lib.tq_matmul_static_ws(None, None, None, rows, cols, ntok, None) == \
            tq.TQ_ERR_WORKSPACE
    assert lib.tq_matmul_static_ws(None, None, None, 1, 100, 9, None) == tq.TQ_ERR_SHAPE
    assert lib.tq_matmul_static_ws(None, None, None, -1, 256, 9, None) == tq.TQ_ERR_SHAPE


def _case(rows, cols, ntok, seed_index):
    s = synth.seeds(seed_index)
    wpq = synth.pq2_0_weights(rows, cols, seed_index)
    x = synth.activations(ntok, cols, s["acts"], s["outliers"])
    return wpq, x


@pytest.mark.gpu
def test_static_workspace_matches_caller_workspace(tq):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gpu_util import DEV, assert_close, gpu_quantize, gpu_repack

    # Calls in a row on the shared array. The first fills whole token tiles
    # (192 = 3 x 64 tokens, no padding), so its data sits where the second
    # call's padded token slots fall: the second (130 tokens, a ragged third
    # tile) must not read any of it. The third (6 tokens, 5120 columns) stages
    # the GEMV's activations in the array over what the others left there.
    # Each result must equal the caller workspace form bit for bit (same
    # kernels, same inputs) and the oracle within the matmul tolerance.
    cases = [(128, 1024, 192, 2), (300, 1024, 130, 3), (100, 5120, 6, 4)]
    assert tq.tq_matmul_workspace_bytes(100, 5120, 6) > 0
    ins, outs = [], []
    for rows, cols, ntok, seed in cases:
        wpq, x = _case(rows, cols, ntok, seed)
        Wtq, Xq = gpu_repack(wpq, rows, cols), gpu_quantize(x)
        Y = torch.full((ntok, rows), float("nan"), dtype=torch.float32, device=DEV)
        tq.tq_matmul_static_ws(Wtq, Xq, Y, rows, cols, ntok)
        ins.append((wpq, x, Wtq, Xq))
        outs.append(Y)
    for (rows, cols, ntok, _), (wpq, x, Wtq, Xq), Y in zip(cases, ins, outs):
        ws = tq.workspace_empty(rows, cols, ntok, DEV)
        ws.fill_(0x5A)
        Yws = torch.full((ntok, rows), float("nan"), dtype=torch.float32, device=DEV)
        tq.tq_matmul_ws(Wtq, Xq, Yws, rows, cols, ntok, ws)
        y_static, y_ws = Y.cpu().numpy(), Yws.cpu().numpy()
        y_ref, abs_sum = oracle.matmul(wpq, oracle.quantize_q8K(x), rows, cols)
        assert np.array_equal(y_static.view(np.uint32), y_ws.view(np.uint32)), \
            f"static and caller workspaces differ at {(rows, cols, ntok)}"
        assert_close(y_static, y_ws, abs_sum)
        assert_close(y_static, y_ref, abs_sum)
    assert tq.tq_device_status() == tq.TQ_OK
