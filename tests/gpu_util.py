"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
call the C ABI through the binding, bring results back as numpy arrays."""
import numpy as np
import torch

import oracle

DEV = "cuda:0"


def ensure_built():
    from bit_matvec_gb300 import build
    build.build()
    oracle.build()


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.uint8).reshape(-1).copy()).to(DEV)


def q8K_from_dev(buf: torch.Tensor, ntok: int, cols: int) -> np.ndarray:
    raw = buf.cpu().numpy()
    return raw.view(oracle.Q8K_DTYPE).reshape(ntok, cols // 256)


def gpu_quantize(x: np.ndarray) -> torch.Tensor:
    import bit_matvec_gb300 as tq
    ntok, cols = x.shape
    X = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)
    Xq = tq.q8K_empty(ntok, cols, DEV)
    tq.tq_quantize_q8K(X, Xq, ntok, cols)
    return Xq


def gpu_repack(wpq: np.ndarray, rows: int, cols: int) -> torch.Tensor:
    import bit_matvec_gb300 as tq
    W = to_dev(wpq)
    Wtq = tq.repacked_empty(rows, cols, DEV)
    tq.tq_repack(W, Wtq, rows, cols)
    return Wtq


def gpu_matmul(Wtq, Xq, rows, cols, ntok) -> np.ndarray:
    import bit_matvec_gb300 as tq
    Y = torch.full((ntok, rows), float("nan"), dtype=torch.float32, device=DEV)
    tq.tq_matmul(Wtq, Xq, Y, rows, cols, ntok)
    return Y.cpu().numpy()


def gpu_groupsums(Wtq, Xq, rows, cols, ntok) -> np.ndarray:
    import bit_matvec_gb300 as tq
    S = torch.full((ntok, rows, cols // 128), -(2 ** 31), dtype=torch.int32, device=DEV)
    tq.tq_matmul_groupsums(Wtq, Xq, S, rows, cols, ntok)
    return S.cpu().numpy()


def assert_close(y_gpu, y_ref, abs_sum, rel=1e-5):
    """|y_gpu - y| <= rel * sum_g |term| (+ a denormal floor), elementwise."""
    assert np.all(np.isfinite(y_gpu))
    err = np.abs(y_gpu.astype(np.float64) - y_ref.astype(np.float64))
    bound = rel * abs_sum + 1e-30
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (f"{len(bad)} outputs out of tolerance, first at {tuple(bad[0])}: "
                           f"gpu {y_gpu[tuple(bad[0])]} ref {y_ref[tuple(bad[0])]} "
                           f"bound {bound[tuple(bad[0])]}")


def gpu_matmul_ws(Wtq, Xq, rows, cols, ntok) -> np.ndarray:
    import bit_matvec_gb300 as tq
    Y = torch.full((ntok, rows), float("nan"), dtype=torch.float32, device=DEV)
    ws = tq.workspace_empty(rows, cols, ntok, DEV)
    ws.fill_(0xAB)   # stale contents must not matter
    tq.tq_matmul_ws(Wtq, Xq, Y, rows, cols, ntok, ws)
    return Y.cpu().numpy()


def gpu_groupsums_ws(Wtq, Xq, rows, cols, ntok) -> np.ndarray:
    import bit_matvec_gb300 as tq
    S = torch.full((ntok, rows, cols // 128), -(2 ** 31), dtype=torch.int32, device=DEV)
    ws = tq.workspace_empty(rows, cols, ntok, DEV)
    ws.fill_(0xCD)
    tq.tq_matmul_groupsums_ws(Wtq, Xq, S, rows, cols, ntok, ws)
    return S.cpu().numpy()
