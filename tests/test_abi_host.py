"""Host-side checks of the C ABI: the library loads, exports every function the
header declares, and rejects bad arguments before touching a GPU.

Fake device addresses are safe here: every rejected call returns before any
CUDA runtime call, and the accepted no-op calls (a zero size) enqueue nothing.
"""
import ctypes

import pytest

import oracle


@pytest.fixture(scope="module")
def lib():
    from bit_matvec_gb300 import build
    build.build()
    import bit_matvec_gb300 as tq
    return tq.library()


def test_exports_every_header_function(lib):
    import bit_matvec_gb300 as tq
    names = tq.header_functions()
    for required in ("tq_quantize_q8K", "tq_repacked_bytes", "tq_repack", "tq_unrepack",
                     "tq_matmul", "tq_matmul_groupsums", "tq_strerror", "tq_matmul_ws",
                     "tq_matmul_workspace_bytes", "tq_matmul_groupsums_ws"):
        assert required in names
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_strerror(lib):
    import bit_matvec_gb300 as tq
    assert tq.tq_version().count(".") == 2
    seen = set()
    for code in (tq.TQ_OK, tq.TQ_ERR_SHAPE, tq.TQ_ERR_NULL, tq.TQ_ERR_ALIGN, tq.TQ_ERR_CUDA,
                 tq.TQ_ERR_TIMEOUT, tq.TQ_ERR_ALIAS, tq.TQ_ERR_WORKSPACE):
        s = tq.tq_strerror(code)
        assert s and s != "unknown error"
        seen.add(s)
    assert len(seen) == 8
    assert tq.tq_strerror(12345) == "unknown error"


@pytest.mark.parametrize("rows,cols", [(32, 256), (100, 512), (1, 128), (32768, 8192),
                                       (17408, 5120), (5120, 17408), (0, 256), (33, 0)])
def test_repacked_bytes_matches_oracle(lib, rows, cols):
    assert lib.tq_repacked_bytes(rows, cols) == oracle.repacked_bytes(rows, cols)
    if rows % 32 == 0:
        assert lib.tq_repacked_bytes(rows, cols) == rows * cols // 128 * 34


def test_repacked_bytes_rejects(lib):
    assert lib.tq_repacked_bytes(32, 100) == -1
    assert lib.tq_repacked_bytes(-1, 256) == -1


A = 0x7F0000000000     # fake, 16-byte aligned device addresses
B = 0x7F1000000000
C = 0x7F2000000000
P = ctypes.c_void_p


def test_shape_errors(lib):
    import bit_matvec_gb300 as tq
    S = tq.TQ_ERR_SHAPE
    assert lib.tq_matmul(P(A), P(B), P(C), 32, 300, 1, None) == S       # cols % 256
    assert lib.tq_matmul(P(A), P(B), P(C), 32, 128, 1, None) == S
    assert lib.tq_matmul(P(A), P(B), P(C), -1, 256, 1, None) == S
    assert lib.tq_matmul(P(A), P(B), P(C), 32, 256, -2, None) == S
    assert lib.tq_matmul_groupsums(P(A), P(B), P(C), 32, 384, 1, None) == S
    assert lib.tq_quantize_q8K(P(A), P(B), 1, 100, None) == S
    assert lib.tq_quantize_q8K(P(A), P(B), -1, 256, None) == S
    assert lib.tq_repack(P(A), P(B), 32, 100, None) == S
    assert lib.tq_unrepack(P(A), P(B), -3, 256, None) == S
    assert lib.tq_repack_ptq1_0(P(A), P(B), 32, 100, None) == S
    assert lib.tq_ptq1_0_bytes(32, 100) == -1
    assert lib.tq_ptq1_0_bytes(-1, 256) == -1
    assert lib.tq_ptq1_0_bytes(3, 256) == 3 * 2 * 28


def test_empty_calls_are_noops(lib):
    import bit_matvec_gb300 as tq
    # no tokens or no rows: nothing to do, even with NULL buffers
    assert lib.tq_matmul(None, None, None, 32, 256, 0, None) == tq.TQ_OK
    assert lib.tq_matmul(None, None, None, 0, 256, 4, None) == tq.TQ_OK
    assert lib.tq_matmul_groupsums(None, None, None, 0, 512, 9, None) == tq.TQ_OK
    assert lib.tq_quantize_q8K(None, None, 0, 256, None) == tq.TQ_OK
    assert lib.tq_quantize_q8K(None, None, 3, 0, None) == tq.TQ_OK
    assert lib.tq_repack(None, None, 0, 256, None) == tq.TQ_OK
    assert lib.tq_unrepack(None, None, 32, 0, None) == tq.TQ_OK
    assert lib.tq_repack_ptq1_0(None, None, 0, 256, None) == tq.TQ_OK


def test_null_errors(lib):
    import bit_matvec_gb300 as tq
    N = tq.TQ_ERR_NULL
    assert lib.tq_matmul(None, P(B), P(C), 32, 256, 1, None) == N
    assert lib.tq_matmul(P(A), None, P(C), 32, 256, 1, None) == N
    assert lib.tq_matmul(P(A), P(B), None, 32, 256, 1, None) == N
    assert lib.tq_matmul(P(A), P(B), None, 32, 0, 1, None) == N          # Y needed to zero it
    assert lib.tq_matmul_groupsums(P(A), P(B), None, 32, 256, 1, None) == N
    assert lib.tq_quantize_q8K(None, P(B), 1, 256, None) == N
    assert lib.tq_quantize_q8K(P(A), None, 1, 256, None) == N
    assert lib.tq_repack(None, P(B), 32, 256, None) == N
    assert lib.tq_unrepack(P(A), None, 32, 256, None) == N
    assert lib.tq_repack_ptq1_0(None, P(B), 32, 256, None) == N


def test_alignment_errors(lib):
    import bit_matvec_gb300 as tq
    E = tq.TQ_ERR_ALIGN
    assert lib.tq_matmul(P(A + 8), P(B), P(C), 32, 256, 1, None) == E     # W needs 16
    assert lib.tq_matmul(P(A), P(B + 4), P(C), 32, 256, 1, None) == E     # Xq needs 16
    assert lib.tq_matmul(P(A), P(B), P(C + 2), 32, 256, 1, None) == E     # Y needs 4
    assert lib.tq_matmul_groupsums(P(A), P(B), P(C + 1), 32, 256, 1, None) == E
    assert lib.tq_quantize_q8K(P(A + 4), P(B), 1, 256, None) == E
    assert lib.tq_quantize_q8K(P(A), P(B + 12), 1, 256, None) == E
    assert lib.tq_repack(P(A + 2), P(B), 32, 256, None) == E
    assert lib.tq_unrepack(P(A), P(B + 8), 32, 256, None) == E
    assert lib.tq_repack_ptq1_0(P(A + 4), P(B), 32, 256, None) == E


def test_alias_errors(lib):
    import bit_matvec_gb300 as tq
    E = tq.TQ_ERR_ALIAS
    wbytes = lib.tq_repacked_bytes(64, 512)
    assert lib.tq_matmul(P(A), P(B), P(A + wbytes - 16), 64, 512, 1, None) == E
    assert lib.tq_matmul(P(A), P(B), P(B + 16), 64, 512, 1, None) == E
    assert lib.tq_quantize_q8K(P(A), P(A + 16), 1, 256, None) == E
    assert lib.tq_repack(P(A), P(A), 32, 256, None) == E                      # in place
    assert lib.tq_unrepack(P(A), P(A + 1088 - 16), 32, 256, None) == E
    assert lib.tq_repack_ptq1_0(P(A), P(A + 32 * 2 * 28 - 16), 32, 256, None) == E


def test_binding_rejects_cpu_tensors(lib):
    import torch
    import bit_matvec_gb300 as tq
    x = torch.zeros(256)
    with pytest.raises(ValueError):
        tq.tq_quantize_q8K(x, torch.zeros(292, dtype=torch.uint8), 1, 256)


def test_workspace_bytes(lib):
    # none for 1..3 tokens; for 4..8 the mma.sync GEMV's staged activations:
    # f16 rows of cols * 2 + 8 bytes (the block's 16-byte multiple), then the
    # half-block sums and the block scales, rounded up to 16 bytes;
    # B tiles + block scales per token tile above
    assert lib.tq_matmul_workspace_bytes(32768, 8192, 1) == 0
    assert lib.tq_matmul_workspace_bytes(32768, 8192, 3) == 0

    def staged(cols, t):
        rows16 = -(-t * (cols * 2 + 8) // 16) * 16
        return -(-(rows16 + t * (cols // 128) * 4 + t * (cols // 256) * 4) // 16) * 16

    for cols, t in ((5120, 4), (5120, 8), (8192, 5), (17408, 4), (9984, 8), (3072, 7)):
        assert lib.tq_matmul_workspace_bytes(17408, cols, t) == staged(cols, t)
    assert lib.tq_matmul_workspace_bytes(17408, 5120, 8) == 83904
    # none below 3072 columns (the fused GEMV is faster there), nor where that
    # GEMV would not fit in a block's 227 KB of shared memory (the larger
    # activations then go to the tensor cores without a workspace)
    for cols, t in ((256, 7), (2816, 4), (10240, 8), (17408, 8), (20224, 4), (1 << 30, 4)):
        assert lib.tq_matmul_workspace_bytes(5120, cols, t) == 0
    # token tiles of 16, 32 and 64: per group 2 x 16 x 128 bytes of B (and per
    # block 3 x 16 floats of scales and sums), 2 x 32 x 128, 2 x 64 x 128
    assert lib.tq_matmul_workspace_bytes(17408, 5120, 9) == 40 * 4096 + 20 * 192
    assert lib.tq_matmul_workspace_bytes(17408, 5120, 16) == 40 * 4096 + 20 * 192
    assert lib.tq_matmul_workspace_bytes(17408, 5120, 17) == 40 * 8192 + 20 * 384
    assert lib.tq_matmul_workspace_bytes(17408, 5120, 33) == 40 * 16384 + 20 * 768
    assert lib.tq_matmul_workspace_bytes(17408, 5120, 64) == 40 * 16384 + 20 * 768
    assert lib.tq_matmul_workspace_bytes(100, 512, 65) == 2 * (4 * 16384 + 2 * 768)
    assert lib.tq_matmul_workspace_bytes(0, 512, 65) == 0
    assert lib.tq_matmul_workspace_bytes(32, 300, 9) == -1
    assert lib.tq_matmul_workspace_bytes(-1, 512, 9) == -1


def test_workspace_errors(lib):
    import bit_matvec_gb300 as tq
    D = 0x7F3000000000
    need = lib.tq_matmul_workspace_bytes(64, 512, 32)
    ws = lib.tq_matmul_ws
    assert ws(P(A), P(B), P(C), 64, 512, 32, None, need, None) == tq.TQ_ERR_NULL
    assert ws(P(A), P(B), P(C), 64, 512, 32, P(D + 8), need, None) == tq.TQ_ERR_ALIGN
    assert ws(P(A), P(B), P(C), 64, 512, 32, P(D), need - 16, None) == tq.TQ_ERR_WORKSPACE
    assert ws(P(A), P(B), P(C), 64, 512, 32, P(C + 64), need, None) == tq.TQ_ERR_ALIAS
    assert ws(P(A), P(B), P(C), 64, 512, 32, P(B), need, None) == tq.TQ_ERR_ALIAS
    assert ws(P(A), P(B), P(C), 64, 300, 32, P(D), need, None) == tq.TQ_ERR_SHAPE
    assert ws(None, None, None, 64, 512, 0, None, 0, None) == tq.TQ_OK
    gs = lib.tq_matmul_groupsums_ws
    assert gs(P(A), P(B), P(C), 64, 512, 32, P(D), need - 1, None) == tq.TQ_ERR_WORKSPACE


def test_matmul_host_errors_before_any_work(lib):
    """tq_matmul_host checks everything its copies and kernels would before it
    enqueues anything, so fake addresses never reach the GPU."""
    import bit_matvec_gb300 as tq
    H, X, D = 0x10000000, 0x7F4000000000, 0x7F3000000000
    f = lib.tq_matmul_host
    need = lib.tq_matmul_workspace_bytes(64, 512, 32)
    args = lambda **k: [P(k.get("w", A)), P(k.get("xh", H)), P(k.get("x", X)), P(k.get("xq", B)),
                        P(k.get("y", C)), P(k.get("yh", H + (1 << 20))), k.get("rows", 64),
                        k.get("cols", 512), k.get("ntok", 32), P(k.get("ws", D)),
                        k.get("wsb", need), None]
    assert f(*args(cols=300)) == tq.TQ_ERR_SHAPE
    assert f(*args(rows=-1)) == tq.TQ_ERR_SHAPE
    assert f(*args(ntok=0)) == tq.TQ_OK
    assert f(*args(xh=0)) == tq.TQ_ERR_NULL
    assert f(*args(yh=0)) == tq.TQ_ERR_NULL
    assert f(*args(x=0)) == tq.TQ_ERR_NULL
    assert f(*args(ws=0)) == tq.TQ_ERR_NULL
    assert f(*args(x=X + 8)) == tq.TQ_ERR_ALIGN
    assert f(*args(y=C + 2)) == tq.TQ_ERR_ALIGN
    assert f(*args(ws=D + 8)) == tq.TQ_ERR_ALIGN
    assert f(*args(wsb=need - 16)) == tq.TQ_ERR_WORKSPACE
    assert f(*args(x=B)) == tq.TQ_ERR_ALIAS
    assert f(*args(y=B)) == tq.TQ_ERR_ALIAS
    assert f(*args(ws=C)) == tq.TQ_ERR_ALIAS
    # one token needs no workspace
    assert f(*args(ntok=1, ws=0, wsb=0, x=0)) == tq.TQ_ERR_NULL


def test_quantize_matmul_errors_before_any_work(lib):
    import bit_matvec_gb300 as tq
    X, D = 0x7F4000000000, 0x7F3000000000
    f = lib.tq_quantize_matmul
    need = lib.tq_matmul_workspace_bytes(64, 512, 32)
    args = lambda **k: [P(k.get("w", A)), P(k.get("x", X)), P(k.get("xq", B)), P(k.get("y", C)),
                        k.get("rows", 64), k.get("cols", 512), k.get("ntok", 32),
                        P(k.get("ws", D)), k.get("wsb", need), None]
    assert f(*args(cols=300)) == tq.TQ_ERR_SHAPE
    assert f(*args(ntok=-1)) == tq.TQ_ERR_SHAPE
    assert f(*args(rows=0)) == tq.TQ_OK
    assert f(*args(x=0)) == tq.TQ_ERR_NULL
    assert f(*args(xq=0)) == tq.TQ_ERR_NULL
    assert f(*args(ws=0)) == tq.TQ_ERR_NULL
    assert f(*args(x=X + 4)) == tq.TQ_ERR_ALIGN
    assert f(*args(xq=B + 8)) == tq.TQ_ERR_ALIGN
    assert f(*args(wsb=need - 1)) == tq.TQ_ERR_WORKSPACE
    assert f(*args(xq=X)) == tq.TQ_ERR_ALIAS
    assert f(*args(y=X + 64)) == tq.TQ_ERR_ALIAS
    assert f(*args(xq=A)) == tq.TQ_ERR_ALIAS
    assert f(*args(ws=X)) == tq.TQ_ERR_ALIAS
    assert f(*args(ntok=1, ws=0, wsb=0, y=0)) == tq.TQ_ERR_NULL
