"""ptq1_0 on the GPU: tq_repack_ptq1_0 decodes the 1.75-bit file into the tq
layout. Its bytes must equal those tq_repack writes for the pq2_0 file of the
same weights, and the oracle's decode-then-repack; products through it match
the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DEV, assert_close, ensure_built, gpu_groupsums, gpu_matmul, gpu_quantize, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _weights(rows, cols, seed):
    s = synth.seeds(seed)
    codes = synth.ternary_codes(rows, cols, s["weights"])
    scales = synth.group_scales(rows, cols, s["scales"])
    sb = np.ascontiguousarray(scales.astype(np.float16)).view(np.uint16)
    return oracle.encode_ptq1_0(codes.astype(np.int8) - 1, sb), synth.pack_pq2_0(codes, scales)


def _repack_ptq1(wpt, rows, cols):
    import bit_matvec_gb300 as tq
    W = to_dev(wpt)
    Wtq = tq.repacked_empty(rows, cols, DEV)
    tq.tq_repack_ptq1_0(W, Wtq, rows, cols)
    return Wtq


@pytest.mark.parametrize("rows,cols", [(32, 128), (100, 256), (300, 1024), (64, 5120)])
def test_repack_ptq1_bit_exact(rows, cols):
    import bit_matvec_gb300 as tq
    wpt, wpq = _weights(rows, cols, 11)
    assert wpt.size == tq.tq_ptq1_0_bytes(rows, cols)
    got = _repack_ptq1(wpt, rows, cols).cpu().numpy()
    W = to_dev(wpq)
    via_pq2 = tq.repacked_empty(rows, cols, DEV)
    tq.tq_repack(W, via_pq2, rows, cols)
    assert np.array_equal(got, via_pq2.cpu().numpy())
    assert np.array_equal(got, oracle.repack(oracle.ptq1_0_to_pq2_0(wpt, rows, cols), rows, cols))


@pytest.mark.parametrize("ntok", [1, 4, 64], ids=lambda t: f"{'tc' if t > 16 else 'gemv'}{t}")
def test_matmul_through_ptq1(ntok):
    rows, cols = 300, 1024
    wpt, _ = _weights(rows, cols, 12)
    x = synth.activations(ntok, cols, synth.seeds(12)["acts"])
    Wtq, Xq = _repack_ptq1(wpt, rows, cols), gpu_quantize(x)
    wpq = oracle.ptq1_0_to_pq2_0(wpt, rows, cols)
    xq = oracle.quantize_q8K(x)
    assert np.array_equal(gpu_groupsums(Wtq, Xq, rows, cols, ntok), oracle.groupsums(wpq, xq, rows, cols))
    y_ref, abs_sum = oracle.matmul(wpq, xq, rows, cols)
    assert_close(gpu_matmul(Wtq, Xq, rows, cols, ntok), y_ref, abs_sum)


def test_repack_ptq1_decode_size():
    """The decode workload's 32768 x 8192 weights as a ptq1_0 file: the whole
    repacked buffer equals tq_repack of the pq2_0 file of the same weights."""
    import bit_matvec_gb300 as tq
    rows, cols = 32768, 8192
    s = synth.seeds(synth.CONFIGS["decode"]["index"])
    codes = synth.ternary_codes(rows, cols, s["weights"])
    scales = synth.group_scales(rows, cols, s["scales"])
    sb = np.ascontiguousarray(scales.astype(np.float16)).view(np.uint16)
    wpt = oracle.encode_ptq1_0(codes.astype(np.int8) - 1, sb)
    a = _repack_ptq1(wpt, rows, cols)
    del wpt
    W = to_dev(synth.pack_pq2_0(codes, scales))
    b = tq.repacked_empty(rows, cols, DEV)
    tq.tq_repack(W, b, rows, cols)
    assert torch.equal(a, b)
