"""IDX_VALIDATE=1: the logits call copies seq_lens and block_tables to the host and refuses a
violated content precondition with IDX_CONTRACT before launching anything; under stream
capture the check is skipped (a device-to-host copy is illegal there) and the call is captured
normally."""
import numpy as np
import pytest
import torch

import oracle
import paged_fp8_mqa_gb300 as idx
from paged_fp8_mqa_gb300 import synth
from gpu_cases import check_logits, expected_row_ends, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture
def validate(monkeypatch):
    monkeypatch.setenv("IDX_VALIDATE", "1")
    idx.device_status(clear=True)
    yield
    assert idx.device_status(clear=True) == 0, "a kernel raised a device status bit"


def _workload():
    return synth.make_workload("validate", 61, 3, 2, 700, "fixed", values=[300, 0, 700])


def _call(w, t, out, bt=None, sl=None):
    idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"] if bt is None else bt,
                   t["seq_lens"] if sl is None else sl, w.max_seq_len, out=out)


def test_valid_inputs_pass(validate):
    w = _workload()
    t = to_device(w)
    out = torch.full((w.rows, idx.idx_padded_seq_len(w.max_seq_len)), float("nan"),
                     device=t["q"].device)
    _call(w, t, out)
    torch.cuda.synchronize()
    ref, tol = oracle.paged_logits(w.q, w.kv_fused, w.weights, w.block_tables, w.seq_lens,
                                   w.max_seq_len, block_size=w.block_size)
    check_logits(w, out, ref, tol)


def test_seq_len_above_max_is_refused(validate):
    w = _workload()
    t = to_device(w)
    out = torch.full((w.rows, idx.idx_padded_seq_len(w.max_seq_len)), 7.0, device=t["q"].device)
    bad = t["seq_lens"].clone()
    bad[1] = w.max_seq_len + 1
    with pytest.raises(idx.IdxError) as e:
        _call(w, t, out, sl=bad)
    assert e.value.status == idx.IDX_CONTRACT and "max_seq_len" in str(e.value)
    torch.cuda.synchronize()
    assert (out == 7.0).all(), "something was launched after IDX_CONTRACT"


def test_out_of_pool_page_is_refused(validate):
    w = _workload()
    t = to_device(w)
    out = torch.full((w.rows, idx.idx_padded_seq_len(w.max_seq_len)), 7.0, device=t["q"].device)
    for bad_id in (w.num_blocks, -1):
        bt = t["bt"].clone()
        bt[2, 5] = bad_id  # request 2 (700 tokens) reads pages 0..10
        with pytest.raises(idx.IdxError) as e:
            _call(w, t, out, bt=bt)
        assert e.value.status == idx.IDX_CONTRACT and "outside the pool" in str(e.value)
    # An out-of-pool entry past a request's own page count is never read: accepted.
    bt = t["bt"].clone()
    bt[0, 10] = w.num_blocks + 5  # request 0 (300 tokens) reads pages 0..4 only
    _call(w, t, out, bt=bt)
    torch.cuda.synchronize()
    assert (out[0:2, :300] != 7.0).all()


def test_skipped_under_capture(validate):
    w = _workload()
    t = to_device(w)
    out = torch.full((w.rows, idx.idx_padded_seq_len(w.max_seq_len)), float("nan"),
                     device=t["q"].device)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _call(w, t, out)  # eager warm-up (and a validated call)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _call(w, t, out)
    g.replay()
    torch.cuda.synchronize()
    ref, tol = oracle.paged_logits(w.q, w.kv_fused, w.weights, w.block_tables, w.seq_lens,
                                   w.max_seq_len, block_size=w.block_size)
    check_logits(w, out, ref, tol)
