"""GB300 (sm_103a) sparse-attention indexer: paged FP8 MQA logits and threshold top-k select.

A thin ctypes binding over ``libidx.so`` (declared in ``include/idx.h``).  It only marshals
arguments: every step of the indexer runs in the library's CUDA kernels, and there is no CPU
fallback -- if the library has not been built, every call raises.

Low-level names mirror the C ABI (``idx_logits_fp8``, ``idx_threshold_select``,
``idx_indexer_threshold_select``, ``idx_schedule``, ``idx_padded_seq_len``,
``idx_min_block_table_width``, ...); they take raw pointers and sizes.  The torch-facing helpers
(``logits_fp8``, ``threshold_select``, ``indexer_threshold_select``, ``schedule``) take tensors,
check dtypes/devices, and pass pointers, strides and the current CUDA stream through.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

_HERE = Path(__file__).resolve().parent
LIB_PATH = _HERE / "libidx.so"

IDX_OK = 0
IDX_INVALID_ARG = 1
IDX_UNSUPPORTED = 2
IDX_CUDA = 3
IDX_CONTRACT = 4
IDX_DTYPE_F32 = 0
IDX_DTYPE_F16 = 1
IDX_DTYPE_BF16 = 2
IDX_DEV_WAIT_TIMEOUT = 1
IDX_DEV_BAD_PAGE = 2
IDX_DEV_INEXACT_SCALE = 4

TILE_TOKENS = 128  # KV positions per work unit of the persistent logits kernel

_lib = None


class IdxError(RuntimeError):
    """A non-zero status from libidx.so."""

    def __init__(self, status: int, message: str):
        super().__init__(f"libidx status {status}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded ``libidx.so``.  Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not LIB_PATH.exists():
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
            "g.build()' or python -m paged_fp8_mqa_gb300.build); the indexer has no CPU path")
    L = ctypes.CDLL(str(LIB_PATH))
    c = ctypes
    P = c.c_void_p
    L.idx_last_error.restype = c.c_char_p
    L.idx_last_error.argtypes = []
    L.idx_padded_seq_len.restype = c.c_int64
    L.idx_padded_seq_len.argtypes = [c.c_int64]
    L.idx_min_block_table_width.restype = c.c_int64
    L.idx_min_block_table_width.argtypes = [c.c_int64, c.c_int32]
    L.idx_num_sms.restype = c.c_int
    L.idx_num_sms.argtypes = [P]
    L.idx_schedule.restype = c.c_int
    L.idx_schedule.argtypes = [P, c.c_int64, c.c_int32, c.c_int32, c.c_int32, P, P]
    L.idx_logits_fp8.restype = c.c_int
    L.idx_logits_fp8.argtypes = [P, P, c.c_int64, c.c_int32, P, P, c.c_int64, c.c_int32, P,
                                 c.c_int64, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
                                 c.c_int32, P, c.c_int32, c.c_int32, P, c.c_int64, P, P]
    L.idx_threshold_select.restype = c.c_int
    L.idx_threshold_select.argtypes = [P, c.c_int64, P, c.c_int32, P, P, P, c.c_int32,
                                       c.c_int32, c.c_int32, P, P, P]
    L.idx_indexer_threshold_select.restype = c.c_int
    L.idx_indexer_threshold_select.argtypes = [
        P, P, c.c_int64, c.c_int32, P, P, c.c_int64, c.c_int32, P, c.c_int64, c.c_int32,
        c.c_int32, c.c_int32, c.c_int32, c.c_int32, c.c_int32, P, P, P, c.c_int32, c.c_int32, P,
        P, P, c.c_int64, P]
    L.idx_mxfp4_workspace_bytes.restype = c.c_int64
    L.idx_mxfp4_workspace_bytes.argtypes = [c.c_int64, c.c_int32, c.c_int32, c.c_int32,
                                            c.c_int32, c.c_int32]
    L.idx_logits_mxfp4.restype = c.c_int
    L.idx_logits_mxfp4.argtypes = [P, P, P, c.c_int64, c.c_int32, P, P, c.c_int64, c.c_int32, P,
                                   c.c_int64, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
                                   c.c_int32, c.c_int32, c.c_int32, P, c.c_int64, P, P,
                                   c.c_int64, P]
    L.idx_device_status.restype = c.c_int
    L.idx_device_status.argtypes = [P, c.c_int32]
    L.idx_debug_withhold_first_tile.restype = c.c_int
    L.idx_debug_withhold_first_tile.argtypes = [c.c_int32]
    _lib = L
    return L


def _check(status: int) -> None:
    if status != IDX_OK:
        raise IdxError(status, lib().idx_last_error().decode())


# ---- C-ABI mirrors (raw pointers / ints) -------------------------------------------------------

def idx_last_error() -> str:
    return lib().idx_last_error().decode()


def idx_padded_seq_len(max_seq_len: int) -> int:
    return int(lib().idx_padded_seq_len(max_seq_len))


def idx_min_block_table_width(seq_len: int, block_size: int) -> int:
    return int(lib().idx_min_block_table_width(seq_len, block_size))


def idx_num_sms() -> int:
    out = ctypes.c_int32(0)
    _check(lib().idx_num_sms(ctypes.byref(out)))
    return out.value


def idx_schedule(seq_lens, seq_lens_stride, batch, next_n, num_sms, schedule, stream) -> int:
    return lib().idx_schedule(seq_lens, seq_lens_stride, batch, next_n, num_sms, schedule, stream)


def idx_logits_fp8(q, kv_fused, num_blocks, block_size, weights, block_tables, bt_row_stride,
                   bt_width, seq_lens, seq_lens_stride, batch, next_n, num_heads, head_dim,
                   max_seq_len, schedule, num_sms, output_dtype, out, out_row_stride,
                   row_ends_out, stream) -> int:
    return lib().idx_logits_fp8(q, kv_fused, num_blocks, block_size, weights, block_tables,
                                bt_row_stride, bt_width, seq_lens, seq_lens_stride, batch, next_n,
                                num_heads, head_dim, max_seq_len, schedule, num_sms,
                                output_dtype, out, out_row_stride, row_ends_out, stream)


def idx_threshold_select(logits, logits_row_stride, row_ends, rows, thresholds, counters,
                         candidates, top_k, capacity, max_context, arrivals, ranges,
                         stream) -> int:
    return lib().idx_threshold_select(logits, logits_row_stride, row_ends, rows, thresholds,
                                      counters, candidates, top_k, capacity, max_context,
                                      arrivals, ranges, stream)


def idx_threshold_select_static(logits, logits_row_stride, row_ends, rows, thresholds,
                                counters, candidates, top_k, capacity, max_context, ranges,
                                stream) -> int:
    """Mirror of the allocation-free select: like idx_threshold_select with repair, but the
    arrival counters live in the library's static device array (at most
    IDX_STATIC_SELECT_MAX_ROWS rows), for callers that cannot allocate a workspace."""
    L = lib()
    f = L.idx_threshold_select_static
    if f.argtypes is None:
        c = ctypes
        f.restype = c.c_int
        f.argtypes = [c.c_void_p, c.c_int64, c.c_void_p, c.c_int32, c.c_void_p, c.c_void_p,
                      c.c_void_p, c.c_int32, c.c_int32, c.c_int32, c.c_void_p, c.c_void_p]
    return f(logits, logits_row_stride, row_ends, rows, thresholds, counters, candidates, top_k,
             capacity, max_context, ranges, stream)


IDX_STATIC_SELECT_MAX_ROWS = 16384
IDX_SELECT_MAX_CONTEXT = 65535 * 8192


def idx_indexer_threshold_select(q, kv_fused, num_blocks, block_size, weights, block_tables,
                                 bt_row_stride, bt_width, seq_lens, seq_lens_stride, batch,
                                 next_n, num_heads, head_dim, max_seq_len, num_sms, thresholds,
                                 counters, candidates, top_k, capacity, arrivals, ranges,
                                 scratch, scratch_row_stride, stream) -> int:
    return lib().idx_indexer_threshold_select(
        q, kv_fused, num_blocks, block_size, weights, block_tables, bt_row_stride, bt_width,
        seq_lens, seq_lens_stride, batch, next_n, num_heads, head_dim, max_seq_len, num_sms,
        thresholds, counters, candidates, top_k, capacity, arrivals, ranges, scratch,
        scratch_row_stride, stream)


def idx_mxfp4_workspace_bytes(num_blocks, block_size, batch, next_n, num_heads,
                              head_dim) -> int:
    return int(lib().idx_mxfp4_workspace_bytes(num_blocks, block_size, batch, next_n, num_heads,
                                               head_dim))


def idx_logits_mxfp4(q, q_sf, kv_fused, num_blocks, block_size, weights, block_tables,
                     bt_row_stride, bt_width, seq_lens, seq_lens_stride, batch, next_n,
                     num_heads, head_dim, max_seq_len, num_sms, output_dtype, out,
                     out_row_stride, row_ends_out, workspace, workspace_bytes, stream) -> int:
    return lib().idx_logits_mxfp4(q, q_sf, kv_fused, num_blocks, block_size, weights,
                                  block_tables, bt_row_stride, bt_width, seq_lens,
                                  seq_lens_stride, batch, next_n, num_heads, head_dim,
                                  max_seq_len, num_sms, output_dtype, out, out_row_stride,
                                  row_ends_out, workspace, workspace_bytes, stream)


def idx_debug_withhold_first_tile(cta: int) -> None:
    _check(lib().idx_debug_withhold_first_tile(int(cta)))


def idx_device_status(clear: bool = False) -> int:
    out = ctypes.c_int32(0)
    _check(lib().idx_device_status(ctypes.byref(out), int(clear)))
    return out.value


# ---- torch-facing marshalling ------------------------------------------------------------------

def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, dims=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {t.dim()}")


def schedule(seq_lens, next_n: int = 1, num_sms: int = 0, out=None, stream=None):
    """The persistent logits kernel's work split, int32 [num_sms + 1, 2] on the device."""
    import torch
    _need(seq_lens, torch.int32, "seq_lens", 1)
    n = num_sms or idx_num_sms()
    if out is None:
        out = torch.empty(n + 1, 2, dtype=torch.int32, device=seq_lens.device)
    _check(idx_schedule(_ptr(seq_lens), seq_lens.stride(0), seq_lens.shape[0], next_n, n,
                        _ptr(out), _stream(stream)))
    return out


def logits_fp8(q, kv_fused, weights, block_tables, seq_lens, max_seq_len: int, *, out=None,
               schedule_meta=None, num_sms: int = 0, row_ends_out=None, stream=None,
               output_dtype=None):
    """Paged FP8 MQA logits.  q: e4m3 (or its uint8 view) [B, next_n, H, D] with H = 8, 16, 32 or 64
    and D = 64 or 128; kv_fused: uint8 whose leading dim is the block count and whose per-block
    bytes are block_size*(D+4) (block_size 32, 64 or 128); weights: float32 [B*next_n, H]; block_tables: int32 [B, W] with unit column stride; seq_lens: int32
    [B] (any stride).  output_dtype: torch.float32 (default) or torch.float16; an `out` buffer
    fixes it.  Returns the [B*next_n, max_seq_len] view of the padded output."""
    import torch
    _need(q, (torch.float8_e4m3fn, torch.uint8), "q", 4)
    _need(kv_fused, torch.uint8, "kv_fused")
    _need(weights, torch.float32, "weights", 2)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, n, H, D = q.shape
    if not q.is_contiguous() or not weights.is_contiguous() or not kv_fused.is_contiguous():
        raise ValueError("q, weights and kv_fused must be contiguous")
    if block_tables.stride(1) != 1:
        raise ValueError("block_tables rows must be contiguous (stride(1) == 1)")
    num_blocks = kv_fused.shape[0]
    block_size = kv_fused.numel() // num_blocks // (D + 4) if num_blocks else 0
    if out is None:
        out = torch.empty(B * n, idx_padded_seq_len(max_seq_len),
                          dtype=output_dtype or torch.float32, device=q.device)
    elif output_dtype is not None and out.dtype != output_dtype:
        raise ValueError(f"out is {out.dtype} but output_dtype is {output_dtype}")
    _need(out, (torch.float32, torch.float16), "out", 2)
    dtype_code = IDX_DTYPE_F16 if out.dtype == torch.float16 else IDX_DTYPE_F32
    if out.stride(1) != 1:
        raise ValueError("out rows must be contiguous")
    _check(idx_logits_fp8(_ptr(q), _ptr(kv_fused), num_blocks, block_size, _ptr(weights),
                          _ptr(block_tables), block_tables.stride(0), block_tables.shape[1],
                          _ptr(seq_lens), seq_lens.stride(0), B, n, H, D, max_seq_len,
                          _ptr(schedule_meta), num_sms, dtype_code, _ptr(out), out.stride(0),
                          _ptr(row_ends_out), _stream(stream)))
    return out[:B * n, :max_seq_len]


def logits_mxfp4(q, q_sf, kv_fused, weights, block_tables, seq_lens, max_seq_len: int, *,
                 out=None, output_dtype=None, workspace=None, num_sms: int = 0,
                 row_ends_out=None, stream=None):
    """MXFP4 paged MQA logits.  q: uint8 [B, next_n, H, D/2] (packed E2M1); q_sf: uint8
    [B, next_n, H, D/32] or its int32 view [B, next_n, H] (UE8M0); kv_fused: uint8 whose leading
    dim is the block count, block_size*(D/2 + D/32) bytes per block; weights float32
    [B*next_n, H]; block_tables, seq_lens as for ``logits_fp8``.  output_dtype: torch.float32
    (the default of this binding, the path checked against the oracle element by element),
    torch.float16, or with head_dim 128 torch.bfloat16 (the pages' default for this variant).
    ``workspace`` (uint8, at least idx_mxfp4_workspace_bytes) is allocated if not given."""
    import torch
    _need(q, torch.uint8, "q", 4)
    _need(q_sf, (torch.uint8, torch.int32), "q_sf")
    _need(kv_fused, torch.uint8, "kv_fused")
    _need(weights, torch.float32, "weights", 2)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, n, H, half = q.shape
    D = 2 * half
    for t, name in ((q, "q"), (q_sf, "q_sf"), (weights, "weights"), (kv_fused, "kv_fused")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q_sf.dtype == torch.int32:
        q_sf = q_sf.view(torch.uint8)
    if q_sf.numel() != B * n * H * (D // 32):
        raise ValueError("q_sf must hold head_dim/32 scale bytes per (b, t, h)")
    if block_tables.stride(1) != 1:
        raise ValueError("block_tables rows must be contiguous (stride(1) == 1)")
    num_blocks = kv_fused.shape[0]
    block_size = kv_fused.numel() // num_blocks // (D // 2 + D // 32) if num_blocks else 0
    if out is None:
        out = torch.empty(B * n, idx_padded_seq_len(max_seq_len),
                          dtype=output_dtype or torch.float32, device=q.device)
    elif output_dtype is not None and out.dtype != output_dtype:
        raise ValueError(f"out is {out.dtype} but output_dtype is {output_dtype}")
    _need(out, (torch.float32, torch.float16, torch.bfloat16), "out", 2)
    need = idx_mxfp4_workspace_bytes(num_blocks, block_size, B, n, H, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _need(workspace, torch.uint8, "workspace")
    dtype_code = {torch.float16: IDX_DTYPE_F16, torch.bfloat16: IDX_DTYPE_BF16}.get(out.dtype,
                                                                                  IDX_DTYPE_F32)
    _check(idx_logits_mxfp4(_ptr(q), _ptr(q_sf), _ptr(kv_fused), num_blocks, block_size,
                            _ptr(weights), _ptr(block_tables), block_tables.stride(0),
                            block_tables.shape[1], _ptr(seq_lens), seq_lens.stride(0), B, n, H, D,
                            max_seq_len, num_sms, dtype_code, _ptr(out), out.stride(0),
                            _ptr(row_ends_out), _ptr(workspace), workspace.numel(),
                            _stream(stream)))
    return out[:B * n, :max_seq_len]


def threshold_select(logits, row_ends, thresholds, counters, candidates, top_k: int,
                     capacity: int, max_context: int, *, arrivals=None, ranges=None,
                     stream=None):
    """Per-row threshold top-k over logits (float32 [rows, >= max_context], unit column stride).
    counters (int32 [rows, 2]) must be zeroed by the caller; candidates is int32
    [rows, top_k + capacity, 2]; arrivals/ranges enable the repair."""
    import torch
    _need(logits, torch.float32, "logits", 2)
    _need(row_ends, torch.int32, "row_ends", 1)
    _need(thresholds, torch.float32, "thresholds", 1)
    _need(counters, torch.int32, "counters", 2)
    _need(candidates, torch.int32, "candidates", 3)
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    rows = row_ends.shape[0]
    for t, name in ((row_ends, "row_ends"), (thresholds, "thresholds"), (counters, "counters"),
                    (candidates, "candidates")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if candidates.shape[1] != top_k + capacity or candidates.shape[0] < rows:
        raise ValueError("candidates must be [rows, top_k + capacity, 2]")
    _check(idx_threshold_select(_ptr(logits), logits.stride(0), _ptr(row_ends), rows,
                                _ptr(thresholds), _ptr(counters), _ptr(candidates), top_k,
                                capacity, max_context, _ptr(arrivals), _ptr(ranges),
                                _stream(stream)))


def indexer_threshold_select(q, kv_fused, weights, block_tables, seq_lens, max_seq_len: int, *,
                             thresholds, counters, candidates, top_k: int, arrivals=None,
                             ranges=None, scratch=None, num_sms: int = 0, stream=None):
    """Scores and threshold select in one pass, without writing the scores.  Inputs as for
    ``logits_fp8``; rows b*next_n + t as there.  thresholds float32 [rows]; counters int32
    [rows, 2] zeroed by the caller; candidates int32 [rows, top_k + capacity, 2].  Passing
    ``arrivals`` (any int32 CUDA tensor; it is not read or written) asks for the repair: every
    row then fits and ``ranges`` (int32 [2, rows]) is written; ``scratch`` (float32
    [rows, >= padded_seq_len]) receives the rescored rows of the requests that need the repair,
    and is allocated here if not given."""
    import torch
    _need(q, (torch.float8_e4m3fn, torch.uint8), "q", 4)
    _need(kv_fused, torch.uint8, "kv_fused")
    _need(weights, torch.float32, "weights", 2)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(thresholds, torch.float32, "thresholds", 1)
    _need(counters, torch.int32, "counters", 2)
    _need(candidates, torch.int32, "candidates", 3)
    B, n, H, D = q.shape
    rows = B * n
    if not q.is_contiguous() or not weights.is_contiguous() or not kv_fused.is_contiguous():
        raise ValueError("q, weights and kv_fused must be contiguous")
    if block_tables.stride(1) != 1:
        raise ValueError("block_tables rows must be contiguous (stride(1) == 1)")
    for t, name in ((thresholds, "thresholds"), (counters, "counters"),
                    (candidates, "candidates")):
        if not t.is_contiguous() or t.shape[0] < rows:
            raise ValueError(f"{name} must be contiguous with at least {rows} rows")
    capacity = candidates.shape[1] - top_k
    if capacity < 0 or candidates.shape[2] != 2:
        raise ValueError("candidates must be [rows, top_k + capacity, 2]")
    if arrivals is not None:
        _need(arrivals, torch.int32, "arrivals", 1)
        if ranges is None:
            raise ValueError("ranges is required with arrivals")
        _need(ranges, torch.int32, "ranges", 2)
        if scratch is None:
            scratch = torch.empty(rows, idx_padded_seq_len(max_seq_len), dtype=torch.float32,
                                  device=q.device)
        _need(scratch, torch.float32, "scratch", 2)
        if scratch.stride(1) != 1:
            raise ValueError("scratch rows must be contiguous")
    num_blocks = kv_fused.shape[0]
    block_size = kv_fused.numel() // num_blocks // (D + 4) if num_blocks else 0
    _check(idx_indexer_threshold_select(
        _ptr(q), _ptr(kv_fused), num_blocks, block_size, _ptr(weights), _ptr(block_tables),
        block_tables.stride(0), block_tables.shape[1], _ptr(seq_lens), seq_lens.stride(0), B, n,
        H, D, max_seq_len, num_sms, _ptr(thresholds), _ptr(counters), _ptr(candidates), top_k,
        capacity, _ptr(arrivals), _ptr(ranges), _ptr(scratch),
        scratch.stride(0) if scratch is not None else 0, _stream(stream)))


def device_status(clear: bool = False) -> int:
    """OR of the IDX_DEV_* bits raised by the kernels since the last clear (synchronous)."""
    return idx_device_status(clear)
