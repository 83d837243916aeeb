"""CPU oracle for the sparse-attention indexer -- TEST INFRASTRUCTURE ONLY.

A plain float64 C implementation (``oracle.c``) of what the indexer computes, wrapped with
ctypes.  Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package; the product path never does, and the two share no code.

Sources restated (see ``oracle.c`` for the passage each function follows):
  * "flashinfer.attn_scores" -- fp8_paged_mqa_logits (formula, Note, Parameters, helpers) and
    fp4_paged_mqa_logits (formula, Parameters q, q_sf, kv_fused).
  * "flashinfer.sdsa.indexer_threshold_select" -- description and Parameters.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_LIB = _HERE / "liboracle.so"

OK = 0
BAD_ARG = -1
BAD_PAGE = -2
BAD_COLUMN = -3


def compile_oracle(src: Path = _SRC, out: Path = _LIB, openmp: bool = True) -> Path:
    """Compile ``src`` into the shared library ``out`` with gcc (float semantics untouched:
    no fast-math, no FMA contraction)."""
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", str(src), "-o",
            str(out), "-lm"]
    if openmp:
        r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
        if r.returncode == 0:
            return out
    subprocess.run(base, check=True, capture_output=True, text=True)
    return out


def build() -> Path:
    """Compile the oracle in place (called by ``__graft_entry__.build()`` and on first use)."""
    return compile_oracle()


_lib_cache: dict[str, ctypes.CDLL] = {}


def load(path: Path | str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library, or another build of ``oracle.c``."""
    key = str(path or _LIB)
    if key in _lib_cache:
        return _lib_cache[key]
    if path is None:
        if not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
            build()
    lib = ctypes.CDLL(key)
    c = ctypes
    P = c.c_void_p
    lib.oracle_e4m3_to_double.restype = c.c_double
    lib.oracle_e4m3_to_double.argtypes = [c.c_uint8]
    lib.oracle_f32_le.restype = c.c_double
    lib.oracle_f32_le.argtypes = [P]
    lib.oracle_min_block_table_width.restype = c.c_int64
    lib.oracle_min_block_table_width.argtypes = [c.c_int64, c.c_int64]
    lib.oracle_padded_seq_len.restype = c.c_int64
    lib.oracle_padded_seq_len.argtypes = [c.c_int64]
    lib.oracle_row_end.restype = c.c_int64
    lib.oracle_row_end.argtypes = [c.c_int64, c.c_int64, c.c_int64]
    lib.oracle_paged_logits.restype = c.c_int
    lib.oracle_paged_logits.argtypes = [P, P, c.c_int64, c.c_int, P, P, c.c_int64, c.c_int64, P,
                                        c.c_int64, c.c_int, c.c_int, c.c_int, c.c_int, P,
                                        c.c_int64, c.c_int64, P, c.c_int]
    lib.oracle_e2m1_to_double.restype = c.c_double
    lib.oracle_e2m1_to_double.argtypes = [c.c_uint8]
    lib.oracle_ue8m0_to_double.restype = c.c_double
    lib.oracle_ue8m0_to_double.argtypes = [c.c_uint8]
    lib.oracle_paged_logits_mxfp4.restype = c.c_int
    lib.oracle_paged_logits_mxfp4.argtypes = [P, P, P, c.c_int64, c.c_int, P, P, c.c_int64,
                                              c.c_int64, P, c.c_int64, c.c_int, c.c_int, c.c_int,
                                              c.c_int, P, c.c_int64, c.c_int64, P, c.c_int]
    lib.oracle_total_order_cmp.restype = c.c_int
    lib.oracle_total_order_cmp.argtypes = [c.c_float, c.c_float]
    lib.oracle_topk.restype = c.c_int
    lib.oracle_topk.argtypes = [P, c.c_int64, P, c.c_int, c.c_int, P, P, c.c_int]
    lib.oracle_select_classify.restype = c.c_int
    lib.oracle_select_classify.argtypes = [P, c.c_int64, P, c.c_int, P, c.c_int, c.c_int, P, P,
                                           P]
    lib.oracle_slot_of.restype = c.c_int64
    lib.oracle_slot_of.argtypes = [c.c_int, c.c_int64, c.c_int, c.c_int]
    lib.oracle_schedule.restype = c.c_int
    lib.oracle_schedule.argtypes = [P, c.c_int64, c.c_int, c.c_int, c.c_int, P]
    lib.oracle_max_threads.restype = c.c_int
    lib.oracle_max_threads.argtypes = []
    _lib_cache[key] = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _np(t):
    """A contiguous numpy view of a CPU torch tensor or numpy array (no copy when possible)."""
    if hasattr(t, "detach"):
        t = t.detach().cpu().contiguous()
        return t.numpy()
    return np.ascontiguousarray(t)


class OracleError(RuntimeError):
    pass


def e4m3_to_double(code: int, lib=None) -> float:
    return (lib or load()).oracle_e4m3_to_double(int(code) & 0xFF)


def f32_le(four_bytes: bytes, lib=None) -> float:
    buf = np.frombuffer(bytes(four_bytes), dtype=np.uint8).copy()
    return (lib or load()).oracle_f32_le(_ptr(buf))


def min_block_table_width(seq_len: int, block_size: int, lib=None) -> int:
    return int((lib or load()).oracle_min_block_table_width(seq_len, block_size))


def padded_seq_len(max_seq_len: int, lib=None) -> int:
    return int((lib or load()).oracle_padded_seq_len(max_seq_len))


def row_end(seq_len: int, next_n: int, t: int, lib=None) -> int:
    return int((lib or load()).oracle_row_end(seq_len, next_n, t))


def row_ends(seq_lens, next_n: int, lib=None) -> np.ndarray:
    """int32 [batch*next_n]: oracle_row_end of every (request, draft slot), row b*next_n + t
    ("flashinfer.attn_scores", fp8_paged_mqa_logits, Note and Returns: slot t of request b
    sees positions 0 .. seq_lens[b] - next_n + t)."""
    lib = lib or load()
    sl = _np(seq_lens).astype(np.int64, copy=False).reshape(-1)
    return np.array([lib.oracle_row_end(int(L), next_n, t) for L in sl for t in range(next_n)],
                    dtype=np.int32)


def paged_logits(q_u8, kv_fused_u8, weights, block_tables, seq_lens, max_seq_len: int,
                 *, block_size: int, out_cols: int | None = None, fill=np.nan,
                 with_tol: bool = True, nthreads: int = 0, lib=None):
    """Float64 logits and tolerance magnitudes.

    q_u8: uint8 [B, next_n, H, D] (e4m3 bytes); kv_fused_u8: uint8 [num_blocks, ...] whose rows
    are block_size*(D+4) bytes; weights: float32 [B*next_n, H]; block_tables: int32 [B, W]
    (row stride taken from the array); seq_lens: int32 [B] (1-D, any stride of a numpy view).
    Returns (logits, tol), float64 [B*next_n, out_cols], entries outside extents = ``fill``.
    """
    lib = lib or load()
    q = _np(q_u8)
    kv = _np(kv_fused_u8)
    w = _np(weights).astype(np.float32, copy=False)
    bt = _np(block_tables).astype(np.int32, copy=False)
    sl = _np(seq_lens).astype(np.int32, copy=False)
    B, n, H, D = q.shape
    num_blocks = kv.shape[0]
    assert kv.reshape(num_blocks, -1).shape[1] == block_size * (D + 4), "kv_fused block size"
    cols = out_cols if out_cols is not None else padded_seq_len(max_seq_len, lib)
    out = np.full((B * n, cols), fill, dtype=np.float64)
    tol = np.full((B * n, cols), fill, dtype=np.float64) if with_tol else None
    st = lib.oracle_paged_logits(_ptr(q), _ptr(kv), num_blocks, block_size, _ptr(w), _ptr(bt),
                                 bt.shape[1], bt.shape[1], _ptr(sl), 1, B, n, H, D, _ptr(out),
                                 cols, cols, _ptr(tol) if with_tol else None, nthreads)
    if st != OK:
        raise OracleError(f"oracle_paged_logits returned {st}")
    return out, tol


def e2m1_to_double(nibble: int, lib=None) -> float:
    return float((lib or load()).oracle_e2m1_to_double(nibble))


def ue8m0_to_double(e: int, lib=None) -> float:
    return float((lib or load()).oracle_ue8m0_to_double(e))


def paged_logits_mxfp4(q_u8, q_sf_u8, kv_fused_u8, weights, block_tables, seq_lens,
                       max_seq_len: int, *, block_size: int, out_cols: int | None = None,
                       fill=np.nan, with_tol: bool = True, nthreads: int = 0, lib=None):
    """Float64 MXFP4 logits and tolerance magnitudes.

    q_u8: uint8 [B, next_n, H, D/2] (packed E2M1); q_sf_u8: uint8 [B, next_n, H, D/32] (UE8M0);
    kv_fused_u8: uint8 [num_blocks, ...] whose rows are block_size*(D/2 + D/32) bytes; weights:
    float32 [B*next_n, H]; block_tables int32 [B, W]; seq_lens int32 [B].
    Returns (logits, tol), float64 [B*next_n, out_cols], entries outside extents = ``fill``.
    """
    lib = lib or load()
    q = _np(q_u8)
    qsf = _np(q_sf_u8)
    kv = _np(kv_fused_u8)
    w = _np(weights).astype(np.float32, copy=False)
    bt = _np(block_tables).astype(np.int32, copy=False)
    sl = _np(seq_lens).astype(np.int32, copy=False)
    B, n, H, half = q.shape
    D = 2 * half
    assert qsf.shape == (B, n, H, D // 32), "q_sf shape"
    num_blocks = kv.shape[0]
    assert kv.reshape(num_blocks, -1).shape[1] == block_size * (D // 2 + D // 32), "block size"
    cols = out_cols if out_cols is not None else padded_seq_len(max_seq_len, lib)
    out = np.full((B * n, cols), fill, dtype=np.float64)
    tol = np.full((B * n, cols), fill, dtype=np.float64) if with_tol else None
    st = lib.oracle_paged_logits_mxfp4(_ptr(q), _ptr(qsf), _ptr(kv), num_blocks, block_size,
                                       _ptr(w), _ptr(bt), bt.shape[1], bt.shape[1], _ptr(sl), 1,
                                       B, n, H, D, _ptr(out), cols, cols,
                                       _ptr(tol) if with_tol else None, nthreads)
    if st != OK:
        raise OracleError(f"oracle_paged_logits_mxfp4 returned {st}")
    return out, tol


def topk(logits_f32, row_ends, top_k: int, nthreads: int = 0, lib=None):
    """Exact top-k per row: (indices [rows, top_k] int32 with -1 padding, counts [rows])."""
    lib = lib or load()
    lg = _np(logits_f32).astype(np.float32, copy=False)
    re = _np(row_ends).astype(np.int32, copy=False)
    rows = lg.shape[0]
    idx = np.full((rows, top_k), -1, dtype=np.int32)
    cnt = np.zeros(rows, dtype=np.int32)
    st = lib.oracle_topk(_ptr(lg), lg.shape[1], _ptr(re), rows, top_k, _ptr(idx), _ptr(cnt),
                         nthreads)
    if st != OK:
        raise OracleError(f"oracle_topk returned {st}")
    return idx, cnt


def select_classify(logits_f32, row_ends, thresholds, top_k: int, capacity: int, lib=None):
    """(n_cand, n_tie, fits) per row, by the threshold rule of the select's description."""
    lib = lib or load()
    lg = _np(logits_f32).astype(np.float32, copy=False)
    re = _np(row_ends).astype(np.int32, copy=False)
    th = _np(thresholds).astype(np.float32, copy=False)
    rows = lg.shape[0]
    nc = np.zeros(rows, dtype=np.int32)
    nt = np.zeros(rows, dtype=np.int32)
    fits = np.zeros(rows, dtype=np.int32)
    st = lib.oracle_select_classify(_ptr(lg), lg.shape[1], _ptr(re), rows, _ptr(th), top_k,
                                    capacity, _ptr(nc), _ptr(nt), _ptr(fits))
    if st != OK:
        raise OracleError(f"oracle_select_classify returned {st}")
    return nc, nt, fits.astype(bool)


def slot_of(is_candidate: bool, n: int, top_k: int, capacity: int, lib=None) -> int:
    return int((lib or load()).oracle_slot_of(int(is_candidate), n, top_k, capacity))


def total_order_cmp(a: float, b: float, lib=None) -> int:
    return int((lib or load()).oracle_total_order_cmp(a, b))


def schedule(seq_lens, tile_tokens: int, num_ctas: int, lib=None) -> np.ndarray:
    """The [num_ctas+1, 2] (request, tile) start points of the even split of KV tiles."""
    lib = lib or load()
    sl = _np(seq_lens).astype(np.int32, copy=False)
    out = np.zeros((num_ctas + 1, 2), dtype=np.int32)
    st = lib.oracle_schedule(_ptr(sl), 1, sl.shape[0], tile_tokens, num_ctas, _ptr(out))
    if st != OK:
        raise OracleError(f"oracle_schedule returned {st}")
    return out


def max_threads(lib=None) -> int:
    return int((lib or load()).oracle_max_threads())


if __name__ == "__main__":  # pragma: no cover
    print(build(), file=sys.stderr)
