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


# ---------------------------------------------------------------- the streamed 1.75-bit form

def _stream_tiles_host(wpt, rows, cols):
    """The stream layout by plain reordering of the file's 28-byte blocks:
    tile (rb, g) holds rows 32 rb .. 32 rb + 31 of group g, row after row; rows
    past the matrix are scale 0 and code bytes 0x80."""
    G = cols // 128
    nrb = -(-rows // 32)
    blocks = np.zeros((nrb * 32, G, 28), np.uint8)
    blocks[:, :, 2:] = 0x80
    blocks[:rows] = wpt.reshape(rows, G, 28)
    return blocks.reshape(nrb, 32, G, 28).transpose(0, 2, 1, 3).reshape(-1)


def _repack_stream(wpt, rows, cols):
    import bit_matvec_gb300 as tq
    W = to_dev(wpt)
    Wt1 = torch.empty(tq.tq_ptq1_0_stream_bytes(rows, cols), dtype=torch.uint8, device=DEV)
    tq.tq_repack_ptq1_0_stream(W, Wt1, rows, cols)
    return Wt1


@pytest.mark.parametrize("rows,cols", [(32, 128), (100, 256), (300, 1024)])
def test_stream_tiles_are_the_file_reordered(rows, cols):
    import bit_matvec_gb300 as tq
    wpt, _ = _weights(rows, cols, 13)
    assert tq.tq_ptq1_0_stream_bytes(rows, cols) == -(-rows // 32) * (cols // 128) * 896
    got = _repack_stream(wpt, rows, cols).cpu().numpy()
    assert np.array_equal(got, _stream_tiles_host(wpt, rows, cols))


@pytest.mark.parametrize("rows,cols,ntok", [(32, 256, 1), (100, 512, 2), (300, 1024, 3),
                                             (300, 1024, 8), (64, 5120, 1), (1000, 2048, 5),
                                             (77, 768, 11), (40, 8192, 1)])
def test_stream_groupsums_exact_matmul_close(rows, cols, ntok):
    """The kernel decodes the base-3 bytes itself: its group sums equal the
    oracle's on the decoded weights bit for bit, and its outputs are within the
    matmul tolerance (11 tokens: launches of 8 and 3)."""
    import bit_matvec_gb300 as tq
    wpt, _ = _weights(rows, cols, 14 + ntok)
    x = synth.activations(ntok, cols, synth.seeds(15)["acts"], synth.seeds(15)["outliers"])
    Wt1, Xq = _repack_stream(wpt, rows, cols), gpu_quantize(x)
    wpq = oracle.ptq1_0_to_pq2_0(wpt, rows, cols)
    xq = oracle.quantize_q8K(x)
    S = torch.full((ntok, rows, cols // 128), -(2 ** 31), dtype=torch.int32, device=DEV)
    tq.tq_matmul_ptq1_0_stream_groupsums(Wt1, Xq, S, rows, cols, ntok)
    assert np.array_equal(S.cpu().numpy(), oracle.groupsums(wpq, xq, rows, cols))
    Y = torch.full((ntok, rows), float("nan"), dtype=torch.float32, device=DEV)
    tq.tq_matmul_ptq1_0_stream(Wt1, Xq, Y, rows, cols, ntok)
    y_ref, abs_sum = oracle.matmul(wpq, xq, rows, cols)
    assert_close(Y.cpu().numpy(), y_ref, abs_sum)
    # the same bits as the 2-bit path on the decoded weights
    Y2 = gpu_matmul(_repack_ptq1(wpt, rows, cols), Xq, rows, cols, ntok)
    if ntok <= 3:   # both run the dp4a loop: identical arithmetic
        assert np.array_equal(Y.cpu().numpy().view(np.uint32), Y2.view(np.uint32))
    assert tq.tq_device_status() == tq.TQ_OK


def test_stream_every_byte_value():
    """Code bytes 0..255 (243..255 lie outside a valid file but still decode by
    the page's formula) in every position of a block, against the oracle."""
    import bit_matvec_gb300 as tq
    rows, cols, ntok = 64, 256, 2
    G = cols // 128
    blocks = np.zeros((rows, G, 28), np.uint8)
    rng_bytes = (synth.splitmix64(0x77, 0, rows * G * 26) >> np.uint64(56)).astype(np.uint8)
    blocks[:, :, 2:] = rng_bytes.reshape(rows, G, 26)
    blocks[:2, 0, 2:] = np.arange(2 * 26, dtype=np.uint8).reshape(2, 26) + 230   # 230..255, 0..25
    blocks[:, :, 0:2] = np.frombuffer(np.float16(0.0125).tobytes(), np.uint8)
    wpt = blocks.reshape(-1)
    x = synth.activations(ntok, cols, synth.seeds(16)["acts"])
    Wt1, Xq = _repack_stream(wpt, rows, cols), gpu_quantize(x)
    wpq = oracle.ptq1_0_to_pq2_0(wpt, rows, cols)
    S = torch.empty((ntok, rows, G), dtype=torch.int32, device=DEV)
    tq.tq_matmul_ptq1_0_stream_groupsums(Wt1, Xq, S, rows, cols, ntok)
    assert np.array_equal(S.cpu().numpy(), oracle.groupsums(wpq, oracle.quantize_q8K(x), rows, cols))
