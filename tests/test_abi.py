"""The C ABI: the library loads, exports every symbol include/idx.h declares, and rejects bad
arguments with status codes before touching the GPU."""
import ctypes
import os
import re

import pytest

import oracle
import paged_fp8_mqa_gb300 as idx

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "idx.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(idx_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from paged_fp8_mqa_gb300 import build
    if not idx.LIB_PATH.exists():
        build.build()
    return idx.lib()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"idx_logits_fp8", "idx_threshold_select", "idx_schedule"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in idx.h but not exported"


def test_helpers_match_worked_examples(lib):
    assert idx.idx_padded_seq_len(8000) == 8192
    assert idx.idx_min_block_table_width(8000, 32) == 250
    assert idx.idx_min_block_table_width(3000, 32) == 94
    assert idx.idx_padded_seq_len(-1) == -1 and idx.idx_min_block_table_width(5, 0) == -1
    for m in (0, 1, 255, 256, 257, 1024, 32768, 65536, 131072, 8000):
        assert idx.idx_padded_seq_len(m) == oracle.padded_seq_len(m)
    for s in (0, 1, 63, 64, 65, 8000):
        for b in (32, 64, 128):
            assert idx.idx_min_block_table_width(s, b) == oracle.min_block_table_width(s, b)


P = ctypes.c_void_p
FAKE = P(1 << 20)  # a 16-byte-aligned non-NULL value: never dereferenced on these paths


def _logits_args(**over):
    a = dict(q=FAKE, kv_fused=FAKE, num_blocks=10, block_size=64, weights=FAKE,
             block_tables=FAKE, bt_row_stride=16, bt_width=16, seq_lens=FAKE,
             seq_lens_stride=1, batch=2, next_n=1, num_heads=64, head_dim=128, max_seq_len=1024,
             schedule=None, num_sms=4, output_dtype=idx.IDX_DTYPE_F32, out=FAKE,
             out_row_stride=1024, row_ends_out=None, stream=None)
    a.update(over)
    return a


@pytest.mark.parametrize("over,code", [
    (dict(q=None), idx.IDX_INVALID_ARG),
    (dict(out=None), idx.IDX_INVALID_ARG),
    (dict(batch=-1), idx.IDX_INVALID_ARG),
    (dict(bt_row_stride=8), idx.IDX_INVALID_ARG),
    (dict(out_row_stride=1000), idx.IDX_INVALID_ARG),
    (dict(out_row_stride=1026), idx.IDX_INVALID_ARG),
    (dict(q=P((1 << 20) + 4)), idx.IDX_INVALID_ARG),
    (dict(num_sms=-3), idx.IDX_INVALID_ARG),
    (dict(num_heads=48), idx.IDX_UNSUPPORTED),
    (dict(num_heads=12), idx.IDX_UNSUPPORTED),
    (dict(head_dim=96), idx.IDX_UNSUPPORTED),
    (dict(head_dim=256), idx.IDX_UNSUPPORTED),
    (dict(block_size=48), idx.IDX_UNSUPPORTED),
    (dict(block_size=256), idx.IDX_UNSUPPORTED),
    (dict(next_n=5), idx.IDX_UNSUPPORTED),
    (dict(output_dtype=2), idx.IDX_UNSUPPORTED),
    (dict(output_dtype=-1), idx.IDX_UNSUPPORTED),
    (dict(batch=5000), idx.IDX_UNSUPPORTED),
    (dict(num_blocks=1 << 26), idx.IDX_INVALID_ARG),
])
def test_logits_rejects_bad_arguments(lib, over, code):
    a = _logits_args(**over)
    st = idx.idx_logits_fp8(*a.values())
    assert st == code, idx.idx_last_error()
    assert idx.idx_last_error()


@pytest.mark.parametrize("over,code", [
    (dict(logits=None), idx.IDX_INVALID_ARG),
    (dict(rows=-1), idx.IDX_INVALID_ARG),
    (dict(top_k=0), idx.IDX_INVALID_ARG),
    (dict(capacity=-1), idx.IDX_INVALID_ARG),
    (dict(logits_row_stride=100), idx.IDX_INVALID_ARG),
    (dict(logits_row_stride=1026), idx.IDX_INVALID_ARG),
    (dict(ranges=None), idx.IDX_INVALID_ARG),
    (dict(capacity=10), idx.IDX_INVALID_ARG),
    (dict(candidates=P((1 << 20) + 4)), idx.IDX_INVALID_ARG),
    (dict(max_context=65535 * 8192 + 1, logits_row_stride=65536 * 8192), idx.IDX_INVALID_ARG),
])
def test_select_rejects_bad_arguments(lib, over, code):
    a = dict(logits=FAKE, logits_row_stride=1024, row_ends=FAKE, rows=4, thresholds=FAKE,
             counters=FAKE, candidates=FAKE, top_k=64, capacity=64, max_context=1024,
             arrivals=FAKE, ranges=FAKE, stream=None)
    a.update(over)
    assert idx.idx_threshold_select(*a.values()) == code, idx.idx_last_error()


def _fused_args(**over):
    a = dict(q=FAKE, kv_fused=FAKE, num_blocks=10, block_size=64, weights=FAKE,
             block_tables=FAKE, bt_row_stride=16, bt_width=16, seq_lens=FAKE,
             seq_lens_stride=1, batch=2, next_n=1, num_heads=64, head_dim=128, max_seq_len=1024,
             num_sms=4, thresholds=FAKE, counters=FAKE, candidates=FAKE, top_k=64, capacity=64,
             arrivals=FAKE, ranges=FAKE, scratch=FAKE, scratch_row_stride=1024, stream=None)
    a.update(over)
    return a


@pytest.mark.parametrize("over,code", [
    (dict(q=None), idx.IDX_INVALID_ARG),
    (dict(thresholds=None), idx.IDX_INVALID_ARG),
    (dict(candidates=None), idx.IDX_INVALID_ARG),
    (dict(batch=-1), idx.IDX_INVALID_ARG),
    (dict(top_k=0), idx.IDX_INVALID_ARG),
    (dict(capacity=-1), idx.IDX_INVALID_ARG),
    (dict(capacity=10), idx.IDX_INVALID_ARG),          # < top_k - 1 with arrivals
    (dict(ranges=None), idx.IDX_INVALID_ARG),
    (dict(scratch=None), idx.IDX_INVALID_ARG),
    (dict(scratch_row_stride=1000), idx.IDX_INVALID_ARG),
    (dict(scratch_row_stride=1026), idx.IDX_INVALID_ARG),
    (dict(scratch=P((1 << 20) + 4)), idx.IDX_INVALID_ARG),
    (dict(candidates=P((1 << 20) + 4)), idx.IDX_INVALID_ARG),
    (dict(counters=P((1 << 20) + 4)), idx.IDX_INVALID_ARG),
    (dict(num_sms=-3), idx.IDX_INVALID_ARG),
    (dict(num_heads=48), idx.IDX_UNSUPPORTED),
    (dict(num_heads=16), idx.IDX_UNSUPPORTED),
    (dict(block_size=48), idx.IDX_UNSUPPORTED),
    (dict(next_n=5), idx.IDX_UNSUPPORTED),
    (dict(batch=5000), idx.IDX_UNSUPPORTED),
])
def test_fused_rejects_bad_arguments(lib, over, code):
    a = _fused_args(**over)
    st = idx.idx_indexer_threshold_select(*a.values())
    assert st == code, idx.idx_last_error()
    assert idx.idx_last_error()


def test_fused_accepts_missing_repair_buffers_without_arrivals(lib):
    """Without arrivals neither ranges nor scratch is needed, and capacity may be small: with
    batch 0 the call then succeeds without touching the GPU."""
    a = _fused_args(arrivals=None, ranges=None, scratch=None, scratch_row_stride=0, capacity=0,
                    batch=0)
    assert idx.idx_indexer_threshold_select(*a.values()) == idx.IDX_OK, idx.idx_last_error()


def test_mxfp4_workspace_size(lib):
    up = lambda x: (x + 255) // 256 * 256
    for nb, bs, b, n, h, d in ((10, 64, 2, 1, 64, 128), (7, 32, 3, 4, 32, 64), (1, 128, 0, 2, 64, 64)):
        # head_dim 128: the KV pages are converted on chip, only q and the weights are staged.
        kv = 0 if d == 128 else up(nb * bs * (d + 4))
        want = kv + up(b * n * h * d) + up(b * n * h * 4)
        assert idx.idx_mxfp4_workspace_bytes(nb, bs, b, n, h, d) == want
    assert idx.idx_mxfp4_workspace_bytes(-1, 64, 1, 1, 64, 128) == -1


def _mxfp4_args(**over):
    a = dict(q=FAKE, q_sf=FAKE, kv_fused=FAKE, num_blocks=10, block_size=64, weights=FAKE,
             block_tables=FAKE, bt_row_stride=16, bt_width=16, seq_lens=FAKE,
             seq_lens_stride=1, batch=2, next_n=1, num_heads=64, head_dim=128, max_seq_len=1024,
             num_sms=4, output_dtype=idx.IDX_DTYPE_F32, out=FAKE, out_row_stride=1024,
             row_ends_out=None, workspace=FAKE, workspace_bytes=1 << 30, stream=None)
    a.update(over)
    return a


@pytest.mark.parametrize("over,code", [
    (dict(q_sf=None), idx.IDX_INVALID_ARG),
    (dict(workspace=None), idx.IDX_INVALID_ARG),
    (dict(workspace_bytes=1000), idx.IDX_INVALID_ARG),
    (dict(workspace=P((1 << 20) + 16)), idx.IDX_INVALID_ARG),
    (dict(head_dim=96), idx.IDX_UNSUPPORTED),
    (dict(num_heads=12), idx.IDX_UNSUPPORTED),
    (dict(next_n=5), idx.IDX_UNSUPPORTED),
    (dict(batch=-1), idx.IDX_INVALID_ARG),
])
def test_mxfp4_rejects_bad_arguments(lib, over, code):
    a = _mxfp4_args(**over)
    assert idx.idx_logits_mxfp4(*a.values()) == code, idx.idx_last_error()


def test_schedule_rejects_bad_arguments(lib):
    assert idx.idx_schedule(None, 1, 4, 1, 8, FAKE, None) == idx.IDX_INVALID_ARG
    assert idx.idx_schedule(FAKE, 0, 4, 1, 8, FAKE, None) == idx.IDX_INVALID_ARG
    assert idx.idx_schedule(FAKE, 1, 4, 9, 8, FAKE, None) == idx.IDX_UNSUPPORTED
    assert idx.idx_schedule(FAKE, 1, 4, 1, 2000, FAKE, None) == idx.IDX_INVALID_ARG


def test_binding_constants_match_the_header():
    import re
    from pathlib import Path
    text = (Path(__file__).resolve().parents[1] / "include" / "idx.h").read_text()
    defs = dict(re.findall(r"#define (IDX_\w+) (-?\d+)", text))
    assert {"IDX_DTYPE_F32", "IDX_DTYPE_F16", "IDX_OK", "IDX_UNSUPPORTED"} <= defs.keys()
    for name, value in defs.items():
        if hasattr(idx, name):
            assert getattr(idx, name) == int(value), name
