"""GPU parity against the CPU oracle, through the C ABI.

Bit-exact: q8_K bytes (scales, int8 values, partial sums), repacked bytes,
and every int32 group sum. Within 1e-5 of sum_g |d_w d_x isum| per output:
the f32 results. Sizes span several tiles with ragged tails. tq_matmul runs
the GEMV up to 16 tokens (int8 activations in shared memory above 8) and the
tensor cores above; the workspace forms run the GEMV up to 8 tokens (from 4
on with its activations staged once in the workspace) and the tensor cores
above (token tiles of 16, 32 and 64).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import read_golden
from gpu_util import (DEV, assert_close, ensure_built, gpu_groupsums, gpu_groupsums_ws, gpu_matmul,
                      gpu_matmul_ws, gpu_quantize, gpu_repack, q8K_from_dev, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _weights(rows, cols, seed_index):
    return synth.pq2_0_weights(rows, cols, seed_index)


def _acts(ntok, cols, seed_index, outliers=True):
    s = synth.seeds(seed_index)
    return synth.activations(ntok, cols, s["acts"], s["outliers"] if outliers else None)


def _q8K_equal(a, b):
    assert np.array_equal(a["d"].view(np.uint32), b["d"].view(np.uint32))
    assert np.array_equal(a["qs"], b["qs"])
    assert np.array_equal(a["bsums"], b["bsums"])


# ---------------------------------------------------------------- quantize

@pytest.mark.parametrize("ntok,cols", [(1, 256), (3, 1024), (7, 2304), (64, 5120), (5, 17408)])
def test_quantize_bit_exact(ntok, cols):
    x = _acts(ntok, cols, 10 + ntok)
    got = q8K_from_dev(gpu_quantize(x), ntok, cols)
    _q8K_equal(got, oracle.quantize_q8K(x))


def test_quantize_special_blocks():
    rows = []
    for name in ("q8K_scale_one.txt", "q8K_scale_two.txt"):
        x = np.zeros(256, dtype=np.float32)
        for tok in read_golden(name):
            if tok[0] not in ("d", "bsums"):
                x[int(tok[0])] = np.float32(tok[1])
        rows.append(x)
    rows.append(np.zeros(256, dtype=np.float32))                       # all zero
    one = np.zeros(256, dtype=np.float32); one[77] = -3.25; rows.append(one)
    rows.append(np.full(256, 1e30, dtype=np.float32))                  # extreme magnitude
    rows.append(np.full(256, -7.0, dtype=np.float32))                  # constant
    ints = np.random.default_rng(3).integers(-127, 128, 256).astype(np.float32)
    ints[5] = 127; rows.append(ints)                                   # exact integers
    tiny = np.linspace(-1, 1, 256, dtype=np.float32) * np.float32(1e-30); rows.append(tiny)
    x = np.stack(rows).reshape(1, -1)
    got = q8K_from_dev(gpu_quantize(x), 1, x.shape[1])
    want = oracle.quantize_q8K(x)
    _q8K_equal(got, want)
    assert got["d"][0, 0] == 1.0 and got["d"][0, 1] == 2.0


# ---------------------------------------------------------------- repack

@pytest.mark.parametrize("rows,cols", [(32, 128), (100, 256), (1, 384), (300, 1024), (64, 5120)])
def test_repack_bit_exact_and_roundtrip(rows, cols):
    import bit_matvec_gb300 as tq
    rng = np.random.default_rng(rows + cols)
    b = rng.integers(0, 256, size=rows * cols // 128 * 34, dtype=np.uint8)   # code 3 included
    Wtq = gpu_repack(b, rows, cols)
    assert np.array_equal(Wtq.cpu().numpy(), oracle.repack(b, rows, cols))
    back = torch.empty(b.size, dtype=torch.uint8, device=DEV)
    tq.tq_unrepack(Wtq, back, rows, cols)
    assert np.array_equal(back.cpu().numpy(), b)


# ---------------------------------------------------------------- group sums and matmul

SHAPES = [(32, 256), (100, 512), (300, 768), (128, 1024)]
GEMV_TOKENS = [1, 2, 3, 4, 5, 7, 8, 9, 12, 15, 16]   # one weight pass for all tokens
TC_TOKENS = [17, 31, 33, 63, 64, 65, 130]           # tensor cores, token tile zero-padded
TC_WS_TOKENS = [9, 12, 16, 17, 31, 32, 33, 63, 64, 65, 130]   # tiles of 16, 32, 64


def _check_product(rows, cols, ntok, ws=False):
    wpq = _weights(rows, cols, 20 + rows % 7)
    x = _acts(ntok, cols, 30 + ntok)
    Wtq = gpu_repack(wpq, rows, cols)
    Xq = gpu_quantize(x)
    xq = oracle.quantize_q8K(x)
    gs, mm = (gpu_groupsums_ws, gpu_matmul_ws) if ws else (gpu_groupsums, gpu_matmul)
    S = gs(Wtq, Xq, rows, cols, ntok)
    assert np.array_equal(S, oracle.groupsums(wpq, xq, rows, cols))
    y_ref, abs_sum = oracle.matmul(wpq, xq, rows, cols)
    assert_close(mm(Wtq, Xq, rows, cols, ntok), y_ref, abs_sum)


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("ntok", GEMV_TOKENS)
def test_gemv_groupsums_exact_matmul_close(rows, cols, ntok):
    _check_product(rows, cols, ntok)


@pytest.mark.parametrize("rows,cols,ntok", [(64, 8192, 4), (64, 8192, 8), (96, 16384, 6),
                                             (64, 5120, 5), (100, 5120, 8), (40, 6144, 4),
                                             (64, 17408, 8), (40, 32768, 5), (33, 65536, 3),
                                             (64, 5120, 16), (40, 3072, 11), (64, 8192, 12),
                                             (64, 8192, 16), (64, 17408, 16)])
def test_gemv_wide_rows(rows, cols, ntok):
    """Long rows: from 4 tokens the tensor-core (mma.sync) variant runs while its
    f16 activations fit in shared memory (8 x 8192 do not: the dp4a loop takes
    over); 16384 columns at 6 tokens exercise the largest staged activations;
    5120 and 6144 columns (40 and 48 groups) take three tiles per warp and
    stage, the others two. Where no variant fits all tokens (8 x 17408,
    5 x 32768, 3 x 65536) the GEMV runs once per half of the tokens. 9 to 16
    tokens keep int8 activations in shared memory and take two 8-column MMAs
    per weight fragment (16 x 5120 with two tiles per warp and stage, 12 x 8192
    with one); 16 x 8192 and 16 x 17408 do not fit and split in halves."""
    _check_product(rows, cols, ntok)


@pytest.mark.parametrize("rows,cols,ntok", [(100, 5120, 4), (40, 5120, 8), (64, 6144, 5),
                                             (33, 9984, 8), (40, 19968, 4), (64, 3072, 7),
                                             (64, 4096, 6), (64, 10240, 8), (40, 20224, 4)])
def test_ws_gemv_staged_activations(rows, cols, ntok):
    """4 to 8 tokens through the workspace forms: a staging kernel converts the
    activations once into the GEMV's f16 rows in the workspace (tq_matmul_ws
    from 5120 columns, tq_quantize_matmul from 3072; up to 9984 columns at 8
    tokens, 19968 at 4, beyond which the workspace size is 0 and the calls
    run as without one). The group sums are exact and Y is within tolerance
    of the oracle; the fused call writes the quantizer's q8_K bytes."""
    import bit_matvec_gb300 as tq
    ws_bytes = tq.tq_matmul_workspace_bytes(rows, cols, ntok)
    assert (ws_bytes > 0) == (3072 <= cols <= (9984 if ntok == 8 else 19968))
    _check_product(rows, cols, ntok, ws=True)
    wpq, x = _weights(rows, cols, 20 + rows % 7), _acts(ntok, cols, 30 + ntok)
    Wtq = gpu_repack(wpq, rows, cols)
    X = torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    Xq = tq.q8K_empty(ntok, cols, DEV)
    Y = torch.full((ntok, rows), float("nan"), dtype=torch.float32, device=DEV)
    ws = tq.workspace_empty(rows, cols, ntok, DEV)
    ws.fill_(0xAB)
    tq.tq_quantize_matmul(Wtq, X, Xq, Y, rows, cols, ntok, ws)
    assert torch.equal(Xq, gpu_quantize(x))
    y_ref, abs_sum = oracle.matmul(wpq, oracle.quantize_q8K(x), rows, cols)
    assert_close(Y.cpu().numpy(), y_ref, abs_sum)
    assert tq.tq_device_status() == tq.TQ_OK


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("ntok", TC_TOKENS)
def test_tc_groupsums_exact_matmul_close(rows, cols, ntok):
    _check_product(rows, cols, ntok)


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("ntok", TC_WS_TOKENS)
def test_tc_ws_groupsums_exact_matmul_close(rows, cols, ntok):
    """The workspace form: activations packed once by a pre-pass."""
    _check_product(rows, cols, ntok, ws=True)


@pytest.mark.parametrize("ntok", [1, 4, 8, 9, 16, 17, 64, 65],
                         ids=lambda t: f"{'tc' if t > 16 else 'gemv'}{t}")
def test_exact_integer_mode(ntok):
    """d_w = 1 and d_x = 1 (integer activations with absmax 127 in every block):
    the output is the exact integer product, on both paths."""
    rows, cols = 96, 1024
    rng = np.random.default_rng(ntok)
    w = rng.integers(-1, 2, size=(rows, cols))
    wpq = synth.pack_pq2_0((w + 1).astype(np.uint8), np.ones((rows, cols // 128), np.float16))
    x = rng.integers(-127, 128, size=(ntok, cols)).astype(np.float32)
    x[:, ::256] = 127.0
    Wtq = gpu_repack(wpq, rows, cols)
    Xq = gpu_quantize(x)
    for mm in (gpu_matmul, gpu_matmul_ws):
        y = mm(Wtq, Xq, rows, cols, ntok)
        assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ w.T)
        assert np.array_equal(y, (x.astype(np.int64) @ w.T).astype(np.float32))


@pytest.mark.parametrize("ntok", [1, 8, 16, 64], ids=lambda t: f"{'tc' if t > 16 else 'gemv'}{t}")
def test_extremes(ntok):
    """All u = 2 (w = +1) or all u = 0 against q = +-127: the largest group sums,
    and activation sums of -16256, 0 and +16256 (the e4m3 path splits each q
    into q & 15 and 16 (q >> 4) and subtracts the sum in its epilogue; these
    are the extremes of both), on the plain and the workspace forms."""
    rows, cols = 64, 512
    for code in (0, 2):
        wpq = synth.pack_pq2_0(np.full((rows, cols), code, np.uint8),
                               np.ones((rows, cols // 128), np.float16))
        alt = np.where(np.arange(cols) % 2 == 0, 127.0, -127.0)
        pats = [np.full(cols, -127.0), alt, np.full(cols, 127.0)]
        x = np.stack([pats[t % 3] for t in range(ntok)]).astype(np.float32)
        Wtq, Xq = gpu_repack(wpq, rows, cols), gpu_quantize(x)
        S_ref = oracle.groupsums(wpq, oracle.quantize_q8K(x), rows, cols)
        for gs in (gpu_groupsums, gpu_groupsums_ws):
            S = gs(Wtq, Xq, rows, cols, ntok)
            assert np.array_equal(S, S_ref)
            assert np.abs(S).max() == 16256


def test_empty_and_degenerate():
    import bit_matvec_gb300 as tq
    rows, cols = 64, 512
    Wtq = gpu_repack(_weights(rows, cols, 1), rows, cols)
    Xq = gpu_quantize(_acts(2, cols, 1))
    Y = torch.full((2, rows), 5.0, device=DEV)
    tq.tq_matmul(Wtq, Xq, Y, rows, cols, 0)          # no tokens: Y untouched
    tq.tq_matmul(Wtq, Xq, Y, 0, cols, 2)             # no rows
    assert torch.all(Y == 5.0)
    tq.tq_matmul(Wtq, Xq, Y, rows, 0, 2)             # empty inner dimension: zeros
    assert torch.all(Y == 0.0)
    with pytest.raises(tq.TQError):
        tq.tq_matmul(Wtq, Xq, Y, rows, 300, 2)


def test_deterministic_and_stream():
    rows, cols, ntok = 200, 2048, 5
    wpq, x = _weights(rows, cols, 2), _acts(ntok, cols, 2)
    Wtq, Xq = gpu_repack(wpq, rows, cols), gpu_quantize(x)
    s = torch.cuda.Stream()
    import bit_matvec_gb300 as tq
    ys = []
    for _ in range(2):
        Y = torch.empty((ntok, rows), device=DEV)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            tq.tq_matmul(Wtq, Xq, Y, rows, cols, ntok, stream=s)
        s.synchronize()
        ys.append(Y.cpu().numpy())
    assert np.array_equal(ys[0].view(np.uint32), ys[1].view(np.uint32))
    assert tq.tq_device_status() == tq.TQ_OK


def test_concurrent_streams():
    """Two streams run the fused quantize + matmul at once (GEMV and tensor-core
    routes), each with its own buffers and workspace, several calls deep; every
    result equals the same call run alone."""
    import bit_matvec_gb300 as tq
    rows, cols = 300, 1024
    wpq = _weights(rows, cols, 7)
    Wtq = gpu_repack(wpq, rows, cols)
    cases = [(1, 7), (64, 8), (9, 9), (130, 10)]
    refs, lanes = [], []
    for ntok, seed in cases:
        x = torch.from_numpy(np.ascontiguousarray(_acts(ntok, cols, seed))).to(DEV)
        Xq, Y = tq.q8K_empty(ntok, cols, DEV), torch.empty((ntok, rows), device=DEV)
        ws = tq.workspace_empty(rows, cols, ntok, DEV)
        tq.tq_quantize_matmul(Wtq, x, Xq, Y, rows, cols, ntok, ws)
        torch.cuda.synchronize()
        refs.append((Xq.clone(), Y.clone()))
        lanes.append((x, tq.q8K_empty(ntok, cols, DEV), torch.empty((ntok, rows), device=DEV),
                      tq.workspace_empty(rows, cols, ntok, DEV), ntok))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for rep in range(3):
        for i, (x, Xq, Y, ws, ntok) in enumerate(lanes):
            tq.tq_quantize_matmul(Wtq, x, Xq, Y, rows, cols, ntok, ws, stream=streams[i % 2])
    torch.cuda.synchronize()
    for (Xq_ref, Y_ref), (_, Xq, Y, _, _) in zip(refs, lanes):
        assert torch.equal(Xq, Xq_ref)
        assert torch.equal(Y.view(torch.int32), Y_ref.view(torch.int32))
    assert tq.tq_device_status() == tq.TQ_OK


@pytest.mark.parametrize("rows,cols,ntok", [(300, 1024, 1), (100, 768, 3), (300, 1024, 4),
                                             (64, 8192, 8), (32, 256, 8), (64, 17408, 8),
                                             (40, 17408, 4), (40, 20224, 4),
                                             (128, 1024, 9), (128, 1024, 16), (64, 17408, 16),
                                             (100, 512, 64), (300, 1024, 65), (160, 2048, 130)])
def test_quantize_matmul_equals_separate_calls(rows, cols, ntok):
    """The fused call gives the bits of tq_quantize_q8K + tq_matmul_ws: Xq and Y
    (GEMV with in-CTA quantization up to 3 tokens; from 4 to 8 a staging
    kernel that quantizes X and stages the GEMV's activations, where they fit
    (not at 8 x 17408 nor 4 x 20224); above, one kernel that
    quantizes and packs the workspace, including the zero padding of a
    ragged last token tile, before the tensor-core kernel)."""
    import bit_matvec_gb300 as tq
    wpq, x = _weights(rows, cols, 5), _acts(ntok, cols, 5)
    Wtq = gpu_repack(wpq, rows, cols)
    Xq_ref = gpu_quantize(x)
    y_ref_dev = gpu_matmul_ws(Wtq, Xq_ref, rows, cols, ntok)
    X = torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    Xq = torch.full_like(Xq_ref, 0xEE)
    Y = torch.full((ntok, rows), float("nan"), dtype=torch.float32, device=DEV)
    ws = tq.workspace_empty(rows, cols, ntok, DEV)
    for _ in range(2):   # twice: the second call follows a matmul (weights read early)
        tq.tq_quantize_matmul(Wtq, X, Xq, Y, rows, cols, ntok, ws)
    assert torch.equal(Xq, Xq_ref)
    assert np.array_equal(Y.cpu().numpy().view(np.uint32), y_ref_dev.view(np.uint32))
    y_ref, abs_sum = oracle.matmul(wpq, oracle.quantize_q8K(x), rows, cols)
    assert_close(Y.cpu().numpy(), y_ref, abs_sum)


@pytest.mark.parametrize("ntok", [1, 6, 64])
def test_matmul_host_matches_device_calls(ntok):
    """The host-to-host step gives the bits of quantize + tq_matmul_ws on device."""
    import bit_matvec_gb300 as tq
    rows, cols = 300, 1024
    wpq, x = _weights(rows, cols, 4), _acts(ntok, cols, 4)
    Wtq = gpu_repack(wpq, rows, cols)
    y_dev = gpu_matmul_ws(Wtq, gpu_quantize(x), rows, cols, ntok)
    x_pin = torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    y_pin = torch.full((ntok, rows), float("nan"), dtype=torch.float32).pin_memory()
    X = torch.empty((ntok, cols), dtype=torch.float32, device=DEV)
    Xq = tq.q8K_empty(ntok, cols, DEV)
    Y = torch.empty((ntok, rows), dtype=torch.float32, device=DEV)
    ws = tq.workspace_empty(rows, cols, ntok, DEV)
    tq.tq_matmul_host(Wtq, x_pin, X, Xq, Y, y_pin, rows, cols, ntok, ws)
    torch.cuda.current_stream().synchronize()
    assert np.array_equal(y_pin.numpy().view(np.uint32), y_dev.view(np.uint32))
    y_ref, abs_sum = oracle.matmul(wpq, oracle.quantize_q8K(x), rows, cols)
    assert_close(y_pin.numpy(), y_ref, abs_sum)


# ---------------------------------------------------------------- full-size workloads

@pytest.mark.parametrize("name", ["tiny", "decode", "small_batch", "prefill"])
def test_workload_sampled_rows(name):
    """Full-size workloads in the same launch configuration the benchmark times;
    the oracle recomputes a sample of rows (first, last, and spread)."""
    wpq, x, cfg = synth.workload(name)
    rows, cols, ntok = cfg["rows"], cfg["cols"], cfg["ntok"]
    Wtq, Xq = gpu_repack(wpq, rows, cols), gpu_quantize(x)
    xq = oracle.quantize_q8K(x)
    _q8K_equal(q8K_from_dev(Xq, ntok, cols), xq)
    y = gpu_matmul(Wtq, Xq, rows, cols, ntok)
    S = gpu_groupsums(Wtq, Xq, rows, cols, ntok)
    y_ws = gpu_matmul_ws(Wtq, Xq, rows, cols, ntok)
    S_ws = gpu_groupsums_ws(Wtq, Xq, rows, cols, ntok)
    assert np.array_equal(S_ws, S)
    rng = np.random.default_rng(rows)
    sample = np.unique(np.concatenate([[0, 1, 31, 32, rows - 1],
                                       rng.integers(0, rows, 60)]))
    wsub = oracle.pq2_0_rows(wpq, cols, sample)
    y_ref, abs_sum = oracle.matmul(wsub, xq, len(sample), cols)
    assert_close(y[:, sample], y_ref, abs_sum)
    assert_close(y_ws[:, sample], y_ref, abs_sum)
    assert np.array_equal(S[:, sample, :], oracle.groupsums(wsub, xq, len(sample), cols))
    # the repacked tiles of the sampled rows hold the same bits as pq2_0
    if rows * cols <= 32768 * 8192:
        wtq = Wtq.cpu().numpy()
        assert np.array_equal(wtq[:oracle.repacked_bytes(64, cols)],
                              oracle.repack(wpq[:64 * cols // 128 * 34], 64, cols))


@pytest.mark.parametrize("m,ntok", [(0, 1), (1, 1), (2, 1), (3, 1), (4, 1), (0, 512), (4, 512)],
                         ids=lambda v: str(v))
def test_replay_matrices_sampled_rows(m, ntok):
    """The decode-step replay's matrices (including the 17408-column W_down) at
    1 token (GEMV) and 512 tokens (tensor cores, workspace form), full size, in
    the benchmark's launch configuration; sampled rows against the oracle."""
    wpq, x, rows, cols = synth.replay_matrix(m, ntok)
    Wtq, Xq = gpu_repack(wpq, rows, cols), gpu_quantize(x)
    xq = oracle.quantize_q8K(x)
    y_ws = gpu_matmul_ws(Wtq, Xq, rows, cols, ntok)
    rng = np.random.default_rng(rows + m)
    sample = np.unique(np.concatenate([[0, 127, 128, rows - 1], rng.integers(0, rows, 12)]))
    wsub = oracle.pq2_0_rows(wpq, cols, sample)
    y_ref, abs_sum = oracle.matmul(wsub, xq, len(sample), cols)
    assert_close(y_ws[:, sample], y_ref, abs_sum)
