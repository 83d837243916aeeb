"""The Python binding only marshals: it never computes on the CPU.  Without the library every
call raises, and host tensors are refused before anything is launched (no GPU needed)."""
import subprocess
import sys
import textwrap
from pathlib import Path

import pytest
import torch

import paged_fp8_mqa_gb300 as idx
from paged_fp8_mqa_gb300 import synth

ROOT = Path(__file__).resolve().parents[1]


def test_missing_library_raises():
    """A binding whose library file is absent raises on first use (there is no fallback)."""
    code = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {str(ROOT)!r})
        from pathlib import Path
        import paged_fp8_mqa_gb300 as idx
        idx.LIB_PATH = Path("/nonexistent/libidx.so")
        idx._lib = None
        try:
            idx.idx_padded_seq_len(8000)
        except RuntimeError as e:
            print("raised:", "no CPU path" in str(e))
        else:
            print("did not raise")
    """)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=120)
    assert out.stdout.strip() == "raised: True", out.stdout + out.stderr


def _host_workload():
    w = synth.make_workload("host", 3, 2, 1, 256, "fixed", values=[200, 100], top_k=16,
                            capacity=15)
    return w, synth.make_mxfp4(w)


def test_host_tensors_are_refused():
    """Every torch-facing entry refuses tensors that are not on a CUDA device."""
    w, m = _host_workload()
    rows = w.rows
    with pytest.raises(TypeError, match="CUDA"):
        idx.logits_fp8(w.q, w.kv_fused, w.weights, w.block_tables, w.seq_lens, w.max_seq_len)
    with pytest.raises(TypeError, match="CUDA"):
        idx.logits_mxfp4(m.q, m.q_sf, m.kv_fused, w.weights, w.block_tables, w.seq_lens,
                         w.max_seq_len)
    with pytest.raises(TypeError, match="CUDA"):
        idx.threshold_select(torch.zeros(rows, 256), torch.zeros(rows, dtype=torch.int32),
                             torch.zeros(rows), torch.zeros(rows, 2, dtype=torch.int32),
                             torch.zeros(rows, 31, 2, dtype=torch.int32), 16, 15, 256)
    with pytest.raises(TypeError, match="CUDA"):
        idx.indexer_threshold_select(
            w.q, w.kv_fused, w.weights, w.block_tables, w.seq_lens, w.max_seq_len,
            thresholds=torch.zeros(rows), counters=torch.zeros(rows, 2, dtype=torch.int32),
            candidates=torch.zeros(rows, 31, 2, dtype=torch.int32), top_k=16)
    with pytest.raises(TypeError, match="CUDA"):
        idx.schedule(w.seq_lens)
