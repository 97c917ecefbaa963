"""The read-ceiling probe computes what it claims: the sum of a buffer's
32-bit words modulo 2^32, on sizes with and without a ragged tail past the
probe's eight-loads-per-thread stride, and in both launch forms."""
import numpy as np
import pytest

import synth


@pytest.mark.gpu
@pytest.mark.parametrize("nbytes", [16, 4096, 1_000_000 - 1_000_000 % 16, 71_443_584])
@pytest.mark.parametrize("early", [False, True])
def test_read_sum_exact(nbytes, early):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gpu_util import DEV, ensure_built
    ensure_built()
    import bit_matvec_gb300 as tq
    host = (synth.splitmix64(0x51, 0, nbytes // 4) >> np.uint64(32)).astype(np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).to(DEV)
    out = torch.zeros(1, dtype=torch.int32, device=DEV)
    tq.tq_probe_read_sum(buf, out, early=early)
    want = int(host.astype(np.uint64).sum() % (1 << 32))
    assert int(out.cpu().numpy().view(np.uint32)[0]) == want


def test_read_sum_rejects_bad_sizes():
    from bit_matvec_gb300 import build
    build.build()
    import bit_matvec_gb300 as tq
    lib = tq.library()
    assert lib.tq_probe_read_sum(None, 8, None, 0, None) == tq.TQ_ERR_SHAPE
    assert lib.tq_probe_read_sum(None, -16, None, 0, None) == tq.TQ_ERR_SHAPE
    assert lib.tq_probe_read_sum(None, 16, None, 0, None) == tq.TQ_ERR_NULL
