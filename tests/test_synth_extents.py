"""The input generator's extent arithmetic (used only to count the benchmark's scores) against
the oracle's pinned extents, on every workload's lengths and on the edge lengths."""
import numpy as np
import pytest
import torch

import oracle
from paged_fp8_mqa_gb300 import synth


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


def test_oracle_row_ends_vector_matches_scalar(lib):
    sl = torch.tensor([0, 1, 2, 3, 4, 63, 64, 65, 300, 1000], dtype=torch.int32)
    for n in range(1, 5):
        got = oracle.row_ends(sl, n, lib=lib)
        want = [oracle.row_end(int(L), n, t, lib=lib) for L in sl for t in range(n)]
        assert got.tolist() == want


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_synth_row_ends_equal_oracle(lib, name):
    spec = {"tiny": (synth.tiny, {}), "decode": (synth.decode, {"batch": 8}),
            "mtp": (synth.mtp, {"batch": 4}), "long_select": (synth.long_select,
                                                              {"batch": 2, "seq_len": 4096}),
            "serving": (synth.serving, {"batch": 16})}[name]
    w = spec[0](**spec[1])
    want = oracle.row_ends(w.seq_lens, w.next_n, lib=lib)
    assert (w.row_ends().numpy() == want).all()
    assert w.valid_scores() == int(want.astype(np.int64).sum())


def test_synth_row_ends_edge_lengths(lib):
    for n in range(1, 5):
        w = synth.make_workload("edge", 5, 6, n, 256, "fixed", values=[0, 1, n - 1, n, n + 1, 256])
        assert (w.row_ends().numpy() == oracle.row_ends(w.seq_lens, n, lib=lib)).all()
