"""Comparison helpers shared by the GPU parity tests (GPU result vs the fp64 oracle)."""
from __future__ import annotations

import numpy as np

# Tolerances on S_i: relative, per input dtype, with an absolute floor of 1e-9 * max S (tokens
# whose fp32 attention probability underflows).
SCORE_RTOL = {"f32": 1e-5, "bf16": 2e-3}
OMEGA_RTOL = 1e-5


def assert_scores_close(S_gpu: np.ndarray, S_ref: np.ndarray, dtype: str, what=""):
    rtol = SCORE_RTOL[dtype]
    floor = 1e-9 * float(np.max(np.abs(S_ref))) if S_ref.size else 0.0
    denom = np.maximum(np.abs(S_ref), max(floor, 1e-300))
    rel = np.abs(S_gpu - S_ref) / denom
    bad = np.flatnonzero(rel > rtol)
    assert bad.size == 0, (f"{what}: {bad.size} scores outside rel {rtol}; worst rel "
                           f"{rel.max():.3e} at {int(np.argmax(rel))} (gpu {S_gpu[np.argmax(rel)]!r}, "
                           f"oracle {S_ref[np.argmax(rel)]!r})")


def chunk_scores(S: np.ndarray, sink: int, w: int, chunk: int) -> np.ndarray:
    n = S.size
    mid = S[sink:n - w]
    return mid.reshape(-1, chunk).mean(axis=1)


def assert_kept_matches(kept_gpu: np.ndarray, S_ref: np.ndarray, *, sink, w, chunk, B, rtol,
                        what=""):
    """Kept sets agree exactly except for chunks whose oracle score lies within rtol of the
    (B/chunk)-th largest oracle chunk score."""
    n = S_ref.size
    kept_gpu = np.asarray(kept_gpu)
    mid = n - sink - w
    if mid <= B:
        assert kept_gpu.tolist() == list(range(n)), what
        return
    assert kept_gpu.size == sink + B + w, what
    assert np.all(np.diff(kept_gpu) > 0), f"{what}: kept positions not ascending"
    assert kept_gpu[:sink].tolist() == list(range(sink)), what
    assert kept_gpu[-w:].tolist() == list(range(n - w, n)), what
    body = kept_gpu[sink:sink + B]
    assert np.all((body - sink) % chunk == np.tile(np.arange(chunk), B // chunk)), \
        f"{what}: kept tokens do not form whole chunks"
    chosen = np.zeros(mid // chunk, dtype=bool)
    chosen[(body[::chunk] - sink) // chunk] = True
    C = chunk_scores(S_ref, sink, w, chunk)
    k = B // chunk
    tau = np.sort(C)[::-1][k - 1]
    ambiguous = np.abs(C - tau) <= rtol * abs(tau)
    want = C > tau
    mismatch = np.flatnonzero((chosen != want) & ~ambiguous)
    assert mismatch.size == 0, (f"{what}: {mismatch.size} clear-cut chunks differ "
                                f"(first {mismatch[:5].tolist()}, tau {tau})")
    assert chosen.sum() == k, what


def assert_kept_valid_for_own_scores(kept: np.ndarray, S: np.ndarray, *, sink, w, chunk, B,
                                     what=""):
    """The kept chunks are a top-(B/chunk) set of the given scores (ties may go either way within
    fp32 rounding of the chunk mean)."""
    n = S.size
    mid = n - sink - w
    if mid <= B:
        assert np.asarray(kept).tolist() == list(range(n)), what
        return
    body = np.asarray(kept)[sink:sink + B]
    chosen = np.zeros(mid // chunk, dtype=bool)
    chosen[(body[::chunk] - sink) // chunk] = True
    C = chunk_scores(S.astype(np.float64), sink, w, chunk)
    lo = C[chosen].min()
    hi = C[~chosen].max()
    assert lo >= hi - 1e-6 * max(abs(hi), 1e-30), f"{what}: kept min {lo} < dropped max {hi}"
