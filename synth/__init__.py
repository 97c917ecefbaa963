"""Seeded synthetic inputs for the ternary pq2_0 x q8_K matrix product.

This module only *draws* inputs: ternary weights w in {-1, 0, +1}, fp16 group
scales, and f32 activations. It writes the weights in the pq2_0 file format,
the input format the method starts from ("ternary bonsai" post, section *what's
running*: 2 bits per weight stored as u = w + 1, one fp16 scale per 128 weights
of a row). It holds none of the method's arithmetic (no quantization, repack or
dot product), so the oracle and the CUDA path can both take their inputs from
here without sharing any of the computation under test.

Random numbers come from splitmix64 (G. Steele, D. Lea, C. Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014), used as a
counter-based generator: value i of the stream with seed s is
mix64(s + (i + 1) * 0x9E3779B97F4A7C15 mod 2^64). Any element can therefore be
regenerated on its own, which lets a test rebuild sampled rows of a
multi-gigabyte workload.

pq2_0 block layout (our reading; the pages give the size, 34 bytes per 128
weights, but not the byte order): little-endian fp16 scale in bytes 0..1, then
32 code bytes; weight k (0..127) of the block sits in code byte k >> 2 at bits
2*(k & 3) .. 2*(k & 3) + 1. Blocks are stored row-major: block (r, g) starts at
byte (r * cols/128 + g) * 34.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

QK_K = 256          # activations per q8_K block
GROUP = 128         # weights per pq2_0 scale
PQ2_BLOCK_BYTES = 34

SEED_BASE = 0x7E570000

# Workloads: (rows, cols, ntok, outlier activations). The sizes and value
# distributions follow the pages' benchmarks (a 32768 x 8192 matvec; a
# 17408 x 5120 weight tile at 4 and 64 tokens) with synthetic data.
CONFIGS = {
    "tiny":        dict(index=0, rows=256,   cols=1024, ntok=1,  outliers=False),
    "decode":      dict(index=1, rows=32768, cols=8192, ntok=1,  outliers=False),
    "small_batch": dict(index=2, rows=17408, cols=5120, ntok=4,  outliers=False),
    "prefill":     dict(index=3, rows=17408, cols=5120, ntok=64, outliers=True),
}

# One transformer block of the decode-step replay: (name, rows, cols).
# The qkv projection is one fused 15360 x 5120 matrix.
REPLAY_BLOCK = (
    ("wqkv", 15360, 5120),
    ("wo", 5120, 5120),
    ("w_gate", 17408, 5120),
    ("w_up", 17408, 5120),
    ("w_down", 5120, 17408),
)
REPLAY_BLOCKS = 64
# Stream seeds of replay matrix m start at SEED_BASE + REPLAY_SEED_OFFSET + 4 m,
# clear of the named workloads' seeds.
REPLAY_SEED_OFFSET = 0x100


def seeds(config_index: int) -> dict:
    """Stream seeds of one workload: weights, scales, activations, outliers."""
    base = SEED_BASE + config_index
    return dict(weights=base, scales=base + 1, acts=base + 2, outliers=base + 3)


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Values start .. start+count-1 of the splitmix64 stream `seed` (uint64)."""
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GOLDEN_GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _chunks(total: int, chunk: int):
    for s in range(0, total, chunk):
        yield s, min(chunk, total - s)


def _parallel_fill(out_flat: np.ndarray, fn, chunk: int) -> None:
    """fn(start, count) -> array of `count` values; written into out_flat."""
    jobs = list(_chunks(out_flat.size, chunk))
    if len(jobs) <= 1:
        for s, n in jobs:
            out_flat[s:s + n] = fn(s, n)
        return
    workers = min(len(jobs), os.cpu_count() or 1, 16)

    def run(job):
        s, n = job
        out_flat[s:s + n] = fn(s, n)

    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(run, jobs))


def ternary_codes(rows: int, cols: int, seed: int, row0: int = 0) -> np.ndarray:
    """u = w + 1 in {0, 1, 2}, each value with probability 1/3 (so p(w=0) = 1/3).

    Element (r, k) uses counter r * cols + k of the stream, so rows
    row0 .. row0+rows-1 of a larger matrix come out identical.
    """
    out = np.empty(rows * cols, dtype=np.uint8)
    base = row0 * cols

    def fn(s, n):
        z = splitmix64(seed, base + s, n)
        return (((z >> np.uint64(32)) * np.uint64(3)) >> np.uint64(32)).astype(np.uint8)

    _parallel_fill(out, fn, 1 << 22)
    return out.reshape(rows, cols)


def group_scales(rows: int, cols: int, seed: int, row0: int = 0,
                 lo: float = 0.005, hi: float = 0.02) -> np.ndarray:
    """fp16 scales drawn U[lo, hi] in f32 and rounded to fp16 (nearest-even).

    Scale (r, g) uses counter r * (cols/128) + g.
    """
    g = cols // GROUP
    z = splitmix64(seed, row0 * g, rows * g)
    u = (z >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    d = np.float32(lo) + np.float32(hi - lo) * u
    return d.astype(np.float16).reshape(rows, g)


def activations(ntok: int, cols: int, seed: int, outlier_seed: int | None = None,
                outlier_p: float = 0.01, outlier_mul: float = 10.0) -> np.ndarray:
    """f32 activations N(0, 1) by Box-Muller (cosine branch), computed in f64.

    Element j = t * cols + k uses counters 2j and 2j+1. With outlier_seed, an
    independent uniform below outlier_p multiplies the element by outlier_mul.
    """
    n = ntok * cols
    out = np.empty(n, dtype=np.float32)

    def fn(s, m):
        z = splitmix64(seed, 2 * s, 2 * m).reshape(m, 2)
        u1 = ((z[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (z[:, 1] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        x = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        if outlier_seed is not None:
            zo = splitmix64(outlier_seed, s, m)
            uo = (zo >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
            x = np.where(uo < outlier_p, x * outlier_mul, x)
        return x.astype(np.float32)

    _parallel_fill(out, fn, 1 << 20)
    return out.reshape(ntok, cols)


def pack_pq2_0(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Write codes u[rows][cols] (0..3) and fp16 scales[rows][cols/128] as pq2_0.

    Returns a flat uint8 array of rows * cols/128 * 34 bytes. Code value 3 is
    not a ternary weight but is written as given (tests use it to show that a
    repack moves bits without interpreting them).
    """
    rows, cols = codes.shape
    assert cols % GROUP == 0 and scales.shape == (rows, cols // GROUP)
    g = cols // GROUP
    c = codes.reshape(rows, g, 32, 4).astype(np.uint8)
    packed = (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)
    sc = np.ascontiguousarray(scales.astype(np.float16)).view(np.uint8).reshape(rows, g, 2)
    return np.concatenate([sc, packed], axis=2).reshape(-1)


def pack_ptq1_0(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Write ternary codes u[rows][cols] (0..2) and fp16 scales as the 1.75-bit
    ptq1_0 file: per 128 weights of a row {fp16 scale; 26 code bytes}, weight
    k in trit k % 5 of code byte k / 5 (the last byte's two spare trits zero),
    and the byte of trits t0..t4 the smallest b with those trits, ceil(256 q /
    243) for q = t0 81 + t1 27 + t2 9 + t3 3 + t4 (the format's encoding; the
    page gives only its decode). Returns a flat uint8 array of rows * cols/128
    * 28 bytes."""
    rows, cols = codes.shape
    assert cols % GROUP == 0 and scales.shape == (rows, cols // GROUP)
    g = cols // GROUP
    t = np.zeros((rows, g, 130), np.int64)
    t[:, :, :GROUP] = codes.reshape(rows, g, GROUP)
    t = t.reshape(rows, g, 26, 5)
    q = t[..., 0] * 81 + t[..., 1] * 27 + t[..., 2] * 9 + t[..., 3] * 3 + t[..., 4]
    packed = ((256 * q + 242) // 243).astype(np.uint8)
    sc = np.ascontiguousarray(scales.astype(np.float16)).view(np.uint8).reshape(rows, g, 2)
    return np.concatenate([sc, packed], axis=2).reshape(-1)


def pq2_0_weights(rows: int, cols: int, config_index: int, row0: int = 0) -> np.ndarray:
    """pq2_0 bytes of rows row0 .. row0+rows-1 of a workload's weight matrix."""
    s = seeds(config_index)
    codes = ternary_codes(rows, cols, s["weights"], row0)
    sc = group_scales(rows, cols, s["scales"], row0)
    return pack_pq2_0(codes, sc)


def replay_seeds(m: int) -> dict:
    """Stream seeds of matrix m of the decode-step replay block."""
    base = SEED_BASE + REPLAY_SEED_OFFSET + 4 * m
    return dict(weights=base, scales=base + 1, acts=base + 2, outliers=base + 3)


def replay_matrix(m: int, ntok: int, row0: int = 0, rows: int | None = None):
    """(pq2_0 bytes of rows row0.., f32 activations[ntok][cols], rows, cols) of
    matrix m of one replay block. Every block of the replay holds a copy of
    these weights in its own allocation."""
    _, nrows, cols = REPLAY_BLOCK[m]
    rows = nrows - row0 if rows is None else rows
    s = replay_seeds(m)
    codes = ternary_codes(rows, cols, s["weights"], row0)
    sc = group_scales(rows, cols, s["scales"], row0)
    x = activations(ntok, cols, s["acts"])
    return pack_pq2_0(codes, sc), x, nrows, cols


def workload(name: str):
    """(pq2_0 bytes, f32 activations[ntok][cols], cfg) of a named workload."""
    cfg = CONFIGS[name]
    s = seeds(cfg["index"])
    w = pq2_0_weights(cfg["rows"], cfg["cols"], cfg["index"])
    x = activations(cfg["ntok"], cfg["cols"], s["acts"],
                    s["outliers"] if cfg["outliers"] else None)
    return w, x, cfg
