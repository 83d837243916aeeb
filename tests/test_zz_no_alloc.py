"""The allocation-free threshold select (idx_threshold_select_static).

It serves callers that cannot allocate device memory -- for example a serving runtime whose
device memory is planned up front with no allocation allowed inside a step, or a plugin with no
access to its host framework's allocator -- and so cannot pass the `arrivals` workspace the
regular select needs.  Here it is called through the C ABI with raw pointers and must return
exactly what the regular entry point returns with a caller-provided workspace, on two calls in
a row (the second reusing the library's static counters the first one left behind).

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_fp8_mqa_gb300 as idx
from paged_fp8_mqa_gb300 import synth
from gpu_cases import (expected_row_ends, expected_scores, check_selection, gpu_logits, gpu_select, kth_values, oracle_logits_cached,
                       selected_from_slots)

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _static_select(logits, row_ends, thresholds, top_k, capacity, max_context):
    rows = row_ends.shape[0]
    d = logits.device
    thr = thresholds.clone().to(d)
    counters = torch.zeros(rows, 2, dtype=torch.int32, device=d)
    cand = torch.full((rows, top_k + capacity, 2), -1, dtype=torch.int32, device=d)
    ranges = torch.full((2, rows), -1, dtype=torch.int32, device=d)
    st = idx.idx_threshold_select_static(
        _ptr(logits), logits.stride(0), _ptr(row_ends), rows, _ptr(thr), _ptr(counters),
        _ptr(cand), top_k, capacity, max_context, _ptr(ranges),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == idx.IDX_OK, idx.idx_last_error()
    torch.cuda.synchronize()
    return dict(thresholds=thr.cpu().numpy(), counters=counters.cpu().numpy(),
                candidates=cand.cpu().numpy(), ranges=ranges.cpu().numpy())


def _selected(logits_cpu, res, row_ends, top_k):
    k = np.minimum(row_ends, top_k)
    return [selected_from_slots(logits_cpu[r], res["candidates"][r], res["ranges"][0, r],
                                res["ranges"][1, r], int(k[r])).tolist()
            for r in range(len(row_ends))]


def test_static_select_matches_workspace_select_on_two_calls():
    idx.device_status(clear=True)
    for name in ("long_select", "serving"):  # two calls in a row, different row counts
        w, ref, _ = oracle_logits_cached(name)
        logits, row_ends = gpu_logits(w, fill=0.0)
        re = expected_row_ends(w)
        kth = torch.from_numpy(kth_values(ref, re, w.top_k))
        thr = (synth.thresholds_below_kth(w, kth) if name == "long_select"
               else synth.thresholds_scaled_kth(w, kth))
        want = gpu_select(logits, row_ends, thr.cuda(), w.top_k, w.capacity, w.max_seq_len)
        got = _static_select(logits, row_ends, thr, w.top_k, w.capacity, w.max_seq_len)
        lc = logits.cpu().numpy()
        # Integer outputs bit-exact, thresholds bit-exact, selections identical.
        assert (got["counters"] == want["counters"]).all()
        assert (got["ranges"] == want["ranges"]).all()
        assert (got["thresholds"].view(np.uint32) == want["thresholds"].view(np.uint32)).all()
        assert _selected(lc, got, re, w.top_k) == _selected(lc, want, re, w.top_k)
        got["arrivals"] = np.zeros(1, dtype=np.int32)  # the static counters are not visible
        check_selection(lc, re, w.top_k, w.capacity, got, thr.numpy())
    assert idx.device_status(clear=True) == 0


def test_static_select_rejects_more_rows_than_its_counters():
    fake = ctypes.c_void_p(1 << 20)
    rows = idx.IDX_STATIC_SELECT_MAX_ROWS + 1
    st = idx.idx_threshold_select_static(fake, 1024, fake, rows, fake, fake, fake, 64, 64, 1024,
                                         fake, None)
    assert st == idx.IDX_INVALID_ARG
    assert str(idx.IDX_STATIC_SELECT_MAX_ROWS) in idx.idx_last_error()
