"""GEMV calls chained back to back in a captured CUDA graph.

Inside a capture, a GEMV that directly follows another GEMV of this library
(no other node between them) and reads nothing that GEMV writes may read its
weights and activations before the earlier one finishes, waiting for it only
before its first store. These tests run such chains, and chains where a call
reads the previous call's output (which must wait), and check that every
output and every q8_K byte equals the same calls run one at a time.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DEV, assert_close, ensure_built, gpu_quantize, gpu_repack

pytestmark = pytest.mark.gpu

# 640 tile columns: at least two per CTA for every GEMV launch shape, the
# condition for the early reads
ROWS = 20480


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _acts(ntok, cols, seed_index):
    s = synth.seeds(seed_index)
    return synth.activations(ntok, cols, s["acts"], s["outliers"])


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(s)
    return g


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t


@pytest.mark.parametrize("rows,cols,ntok", [(ROWS, 1024, 1), (ROWS, 1024, 3), (ROWS, 1024, 4),
                                             (ROWS, 1024, 8), (5120, 17408, 1), (5120, 17408, 3),
                                             (5120, 17408, 4), (32768, 1024, 1), (32768, 1024, 4),
                                             (ROWS, 5120, 8), (ROWS, 3072, 5)])
def test_graph_chain_of_independent_calls(rows, cols, ntok):
    """Four fused calls and two tq_matmul calls, each on its own weights, all
    reading activations no call of the chain writes (the fused calls share
    one q8_K output buffer): the early-read form runs from the second call on.
    With 1024 columns every CTA has several tile columns and waits after its
    first; 5120 x 17408 gives one long tile column per CTA, and the one- and
    three-token kernels wait after its first ring stage. With 32768 rows (1024
    tile columns) the calls made one at a time, which wait first, fill every
    resident slot with uneven tile columns per CTA, while the chain splits
    them evenly over fewer CTAs: the bits must not change. From 4 tokens and
    3072 columns each fused call is a staging kernel and the GEMV, which the
    staging kernel lets start at once (5120 x 17408 at 4 tokens, 20480 x 5120
    at 8, 20480 x 3072 at 5)."""
    import bit_matvec_gb300 as tq
    n = 4
    wpq = [synth.pq2_0_weights(rows, cols, 40 + i) for i in range(n + 2)]
    Ws = [gpu_repack(w, rows, cols) for w in wpq]
    x = _acts(ntok, cols, 41)
    X = torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    Xq_in = gpu_quantize(_acts(ntok, cols, 42))
    ws = tq.workspace_empty(rows, cols, ntok, DEV)

    def run(s, Ys, Xq):
        for i in range(n):
            tq.tq_quantize_matmul(Ws[i], X, Xq, Ys[i], rows, cols, ntok, ws, stream=s)
        for i in range(2):
            tq.tq_matmul(Ws[n + i], Xq_in, Ys[n + i], rows, cols, ntok, stream=s)

    # one call at a time
    refs = []
    Xq_ref = tq.q8K_empty(ntok, cols, DEV)
    for i in range(n + 2):
        Y = torch.empty((ntok, rows), device=DEV)
        if i < n:
            tq.tq_quantize_matmul(Ws[i], X, Xq_ref, Y, rows, cols, ntok, ws)
        else:
            tq.tq_matmul(Ws[i], Xq_in, Y, rows, cols, ntok)
        torch.cuda.synchronize()
        refs.append(Y)
    assert torch.equal(Xq_ref, gpu_quantize(x))

    Ys = [torch.full((ntok, rows), float("nan"), device=DEV) for _ in range(n + 2)]
    Xq = torch.full_like(Xq_ref, 0xEE)
    g = _capture(lambda s: run(s, Ys, Xq))
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        for Y, R in zip(Ys, refs):
            assert torch.equal(_bits(Y), _bits(R))
        assert torch.equal(Xq, Xq_ref)
        for Y in Ys:
            Y.fill_(float("nan"))
        Xq.fill_(0xEE)
    assert tq.tq_device_status() == tq.TQ_OK

    # and against the oracle, for the first and the last weights
    xq = oracle.quantize_q8K(x)
    for i in (0, n - 1):
        rows_s = np.r_[0:64, rows - 64:rows]
        y_ref, abs_sum = oracle.matmul(wpq[i].reshape(rows, -1)[rows_s].reshape(-1), xq,
                                       len(rows_s), cols)
        assert_close(refs[i].cpu().numpy()[:, rows_s], y_ref, abs_sum)


def _wide(wpq, rows, cols, reps):
    """pq2_0 bytes of a rows x (cols * reps) matrix: each row repeated reps times."""
    return np.tile(wpq.reshape(rows, -1), (1, reps)).reshape(-1)


@pytest.mark.parametrize("ntok,n", [(1, ROWS), (4, ROWS), (4, 16384), (8, 8192)])
def test_graph_chain_reading_previous_outputs(ntok, n):
    """Each call reads what the call before it wrote (its Y as the next
    activations, or its q8_K bytes): those calls wait before reading, and the
    results equal the calls run one at a time. One call in the chain reads
    only older outputs and may read early. At 4 tokens and 16384 columns, and 8
    tokens and 8192, the fused calls on the square matrices stage their
    activations in the workspace (a staging kernel, then the GEMV)."""
    import bit_matvec_gb300 as tq
    c0, reps = 1024, n // 1024
    w0 = synth.pq2_0_weights(n, c0, 50)
    W1 = gpu_repack(w0, n, c0)                               # c0 -> n
    W2 = gpu_repack(_wide(synth.pq2_0_weights(n, c0, 51), n, c0, reps), n, n)
    W3 = gpu_repack(_wide(synth.pq2_0_weights(n, c0, 52), n, c0, reps), n, n)
    W4 = gpu_repack(_wide(synth.pq2_0_weights(n, c0, 53), n, c0, reps), n, n)
    X0 = torch.from_numpy(np.ascontiguousarray(_acts(ntok, c0, 54))).to(DEV)
    ws0 = tq.workspace_empty(n, c0, ntok, DEV)
    ws = tq.workspace_empty(n, n, ntok, DEV)

    def buffers():
        return dict(Y1=torch.full((ntok, n), float("nan"), device=DEV),
                    Y2=torch.full((ntok, n), float("nan"), device=DEV),
                    Y3=torch.full((ntok, n), float("nan"), device=DEV),
                    Y4=torch.full((ntok, n), float("nan"), device=DEV),
                    Y5=torch.full((ntok, n), float("nan"), device=DEV),
                    Xq0=torch.full((tq.q8K_nbytes(ntok, c0),), 0xEE, dtype=torch.uint8, device=DEV),
                    Xq1=torch.full((tq.q8K_nbytes(ntok, n),), 0xEE, dtype=torch.uint8, device=DEV),
                    Xq2=torch.full((tq.q8K_nbytes(ntok, n),), 0xEE, dtype=torch.uint8, device=DEV))

    def steps(b):
        return [
            lambda s: tq.tq_quantize_matmul(W1, X0, b["Xq0"], b["Y1"], n, c0, ntok, ws0, stream=s),
            # activations = the previous call's Y
            lambda s: tq.tq_quantize_matmul(W2, b["Y1"], b["Xq1"], b["Y2"], n, n, ntok, ws, stream=s),
            # q8_K bytes the previous call wrote
            lambda s: tq.tq_matmul(W3, b["Xq1"], b["Y3"], n, n, ntok, stream=s),
            # Y of two calls back (complete once the previous call has waited)
            lambda s: tq.tq_quantize_matmul(W4, b["Y2"], b["Xq2"], b["Y4"], n, n, ntok, ws, stream=s),
            # the previous call's Y again
            lambda s: tq.tq_quantize_matmul(W2, b["Y4"], b["Xq1"], b["Y5"], n, n, ntok, ws, stream=s),
        ]

    ref = buffers()
    for step in steps(ref):
        step(torch.cuda.current_stream())
        torch.cuda.synchronize()
    got = buffers()
    g = _capture(lambda s: [step(s) for step in steps(got)])
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(_bits(got[k]), _bits(ref[k])), k
    assert all(torch.isfinite(ref[k]).all() for k in ("Y1", "Y2", "Y3", "Y4", "Y5"))
    assert tq.tq_device_status() == tq.TQ_OK


def test_eager_chain_equals_graph():
    """The same independent chain run eagerly (where calls always wait before
    reading) and captured give the same bits."""
    import bit_matvec_gb300 as tq
    cols, ntok = 2048, 1
    Ws = [gpu_repack(synth.pq2_0_weights(ROWS, cols, 60 + i), ROWS, cols) for i in range(3)]
    X = torch.from_numpy(np.ascontiguousarray(_acts(ntok, cols, 61))).to(DEV)
    ws = tq.workspace_empty(ROWS, cols, ntok, DEV)

    def run(s, Ys, Xq):
        for W, Y in zip(Ws, Ys):
            tq.tq_quantize_matmul(W, X, Xq, Y, ROWS, cols, ntok, ws, stream=s)

    eager = ([torch.empty((ntok, ROWS), device=DEV) for _ in Ws], tq.q8K_empty(ntok, cols, DEV))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(s, *eager)
    s.synchronize()
    graph = ([torch.empty((ntok, ROWS), device=DEV) for _ in Ws], tq.q8K_empty(ntok, cols, DEV))
    g = _capture(lambda st: run(st, *graph))
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager[0], graph[0]):
        assert torch.equal(_bits(a), _bits(b))
    assert torch.equal(eager[1], graph[1])


def test_graph_chain_mixed_kinds_sharing_a_workspace():
    """Staged GEMV calls beside the quantizer and the tensor-core path, all on
    one workspace: a staging kernel after the quantizer (it must wait before
    reading the q8_K bytes), the quantize-and-pack kernel after a staged GEMV
    (it must not rewrite the workspace before that GEMV has loaded it), a
    staging kernel after the tensor-core kernel, and one after a staged GEMV
    (its input final, read before waiting). The staging kernel lets its GEMV
    start at once, so that GEMV may read its weights beside the kernel before
    the staging kernel. Captured and eager runs give the bits of the calls
    made one at a time."""
    import bit_matvec_gb300 as tq
    rows, cols = 8192, 5120
    Ws = [gpu_repack(synth.pq2_0_weights(rows, cols, 70 + i), rows, cols) for i in range(3)]
    X8 = torch.from_numpy(np.ascontiguousarray(_acts(8, cols, 71))).to(DEV)
    X16 = torch.from_numpy(np.ascontiguousarray(_acts(16, cols, 72))).to(DEV)
    nb = max(tq.tq_matmul_workspace_bytes(rows, cols, 8), tq.tq_matmul_workspace_bytes(rows, cols, 16))
    assert tq.tq_matmul_workspace_bytes(rows, cols, 8) > 0
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)

    def buffers():
        return dict(Xq8=tq.q8K_empty(8, cols, DEV), Xq8b=tq.q8K_empty(8, cols, DEV),
                    Xq16=tq.q8K_empty(16, cols, DEV),
                    **{f"Y{i}": torch.full((16 if i == 2 else 8, rows), float("nan"), device=DEV)
                       for i in range(1, 5)})

    def steps(b):
        return [
            lambda s: tq.tq_quantize_q8K(X8, b["Xq8"], 8, cols, stream=s),
            lambda s: tq.tq_matmul_ws(Ws[0], b["Xq8"], b["Y1"], rows, cols, 8, ws, stream=s),
            lambda s: tq.tq_quantize_matmul(Ws[1], X16, b["Xq16"], b["Y2"], rows, cols, 16, ws,
                                            stream=s),
            lambda s: tq.tq_matmul_ws(Ws[2], b["Xq8"], b["Y3"], rows, cols, 8, ws, stream=s),
            lambda s: tq.tq_quantize_matmul(Ws[0], X8, b["Xq8b"], b["Y4"], rows, cols, 8, ws,
                                            stream=s),
        ]

    ref = buffers()
    for step in steps(ref):
        step(torch.cuda.current_stream())
        torch.cuda.synchronize()
    assert torch.equal(_bits(ref["Y1"]), _bits(ref["Y4"]))
    assert torch.equal(ref["Xq8"], ref["Xq8b"])
    eager = buffers()
    for step in steps(eager):
        step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    got = buffers()
    g = _capture(lambda s: [step(s) for step in steps(got)])
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(_bits(got[k]), _bits(ref[k])), k
            assert torch.equal(_bits(eager[k]), _bits(ref[k])), k
    assert tq.tq_device_status() == tq.TQ_OK
    xq = oracle.quantize_q8K(_acts(8, cols, 71))
    rows_s = np.r_[0:32, rows - 32:rows]
    w0 = synth.pq2_0_weights(rows, cols, 70).reshape(rows, -1)
    y_ref, abs_sum = oracle.matmul(w0[rows_s].reshape(-1), xq, len(rows_s), cols)
    assert_close(ref["Y1"].cpu().numpy()[:, rows_s], y_ref, abs_sum)
