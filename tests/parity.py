"""The parity rule for GPU results against the CPU oracle.

A GPU fp16 value g matches the oracle's fp16 value r when
    |g - r| <= 2 * ulp16(r),   or   |r| < 1 and |g - r| <= 1e-3,
with ulp16(r) = 2^(floor(log2 |r|) - 10) for |r| >= 2^-14 and 2^-24 below;
an infinite r must be matched exactly and g must never be NaN.

Why this bound: the oracle rounds the exact sum to fp16 once; the GPU
accumulates in fp32 (about 112 roundings of a K=64 partial sum into the
accumulator at k = 7168, relative error a few 1e-6 -- far below an fp16 ulp)
and then rounds to fp16, so the two can differ by one fp16 rounding step near
a rounding boundary; 2 ulps leaves a factor of two of margin, and the absolute
floor covers cancellation near zero where the fp32 error is relative to the
partial sums, not to C.
"""
import numpy as np


def ulp16(r: np.ndarray) -> np.ndarray:
    a = np.abs(r.astype(np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0 ** -14, np.exp2(e - 10), 2.0 ** -24)


def parity_mask(gpu: np.ndarray, ref: np.ndarray) -> np.ndarray:
    g = np.asarray(gpu, dtype=np.float16).astype(np.float64)
    r = np.asarray(ref, dtype=np.float16).astype(np.float64)
    ok = np.zeros(r.shape, dtype=bool)
    inf = np.isinf(r)
    ok[inf] = g[inf] == r[inf]
    fin = np.isfinite(r) & np.isfinite(g)
    d = np.abs(g - r)
    ok[fin] = (d[fin] <= 2.0 * ulp16(r[fin])) | ((np.abs(r[fin]) < 1.0) & (d[fin] <= 1e-3))
    return ok


def assert_parity(gpu, ref, what: str = "") -> None:
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert not np.isnan(gpu.astype(np.float32)).any(), f"{what}: NaN in GPU result"
    ok = parity_mask(gpu, ref)
    if not ok.all():
        bad = np.argwhere(~ok)
        first = [tuple(int(v) for v in b) for b in bad[:8]]
        vals = [(float(gpu[b]), float(ref[b])) for b in first]
        raise AssertionError(f"{what}: {len(bad)} of {ok.size} outside tolerance; first {first}: {vals}")


def block_samples(rng, m: int, n: int, block: int = 32, per_block: int = 2, edges: bool = True):
    """Output coordinates that reach every `block` x `block` cell of an m x n C:
    `per_block` random (row, col) pairs inside each cell (clipped to the
    matrix), plus, with `edges`, the whole last row and last column (the M and N
    tails). Every (tile, column chunk, TMEM lane quarter) of any tiling whose
    tile sides are multiples of `block` holds at least one sample."""
    rb = -(-m // block)
    cb = -(-n // block)
    r0 = np.repeat(np.arange(rb) * block, cb * per_block)
    c0 = np.tile(np.repeat(np.arange(cb) * block, per_block), rb)
    rows = r0 + rng.integers(0, block, r0.size)
    cols = c0 + rng.integers(0, block, c0.size)
    rows = np.minimum(rows, m - 1)
    cols = np.minimum(cols, n - 1)
    if edges:
        rows = np.concatenate([rows, np.full(n, m - 1), np.arange(m)])
        cols = np.concatenate([cols, np.arange(n), np.full(m, n - 1)])
    return rows.astype(np.int32), cols.astype(np.int32)
