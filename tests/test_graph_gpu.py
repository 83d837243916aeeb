"""The whole serving indexer (counter reset, logits with the in-kernel schedule, threshold
select with repair) captured in one CUDA graph and replayed with new seq_lens contents."""
import numpy as np
import pytest
import torch

import paged_fp8_mqa_gb300 as idx
from paged_fp8_mqa_gb300 import synth
from gpu_cases import (expected_row_ends, expected_scores, check_logits, check_selection, kth_values, oracle_logits_cached,
                       selected_from_slots)

pytestmark = pytest.mark.gpu


def test_serving_indexer_graph_replay():
    w, ref, tol = oracle_logits_cached("serving")
    d = torch.device("cuda:0")
    q, kv, wt = w.q.to(d), w.kv_fused.to(d), w.weights.to(d)
    bt, sl = w.block_tables.to(d), w.seq_lens.to(d)
    rows, pad = w.rows, idx.idx_padded_seq_len(w.max_seq_len)
    kth = torch.from_numpy(kth_values(ref, expected_row_ends(w), w.top_k))
    thr0 = synth.thresholds_scaled_kth(w, kth)
    out = torch.zeros(rows, pad, device=d)
    row_ends = torch.zeros(rows, dtype=torch.int32, device=d)
    thr = thr0.to(d)
    counters = torch.zeros(rows, 2, dtype=torch.int32, device=d)
    cand = torch.zeros(rows, w.top_k + w.capacity, 2, dtype=torch.int32, device=d)
    arrivals = torch.zeros(rows, dtype=torch.int32, device=d)
    ranges = torch.zeros(2, rows, dtype=torch.int32, device=d)

    def step():
        counters.zero_()
        idx.logits_fp8(q, kv, wt, bt, sl, w.max_seq_len, out=out, row_ends_out=row_ends)
        idx.threshold_select(out, row_ends, thr, counters, cand, w.top_k, w.capacity,
                             w.max_seq_len, arrivals=arrivals, ranges=ranges)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()  # eager warm-up loads the kernels before capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    thr.copy_(thr0.to(d))
    with torch.cuda.graph(graph, stream=s):
        step()
    for trial in range(2):
        if trial == 1:
            # New contents for the captured buffers: shorter sequences (their pages stay valid).
            g = torch.Generator().manual_seed(11)
            new = (w.seq_lens.to(torch.float64) * torch.rand(w.batch, generator=g)).to(torch.int32)
            w = synth.Workload(**{**w.__dict__, "seq_lens": new})
            sl.copy_(new.to(d))
            import oracle
            ref, tol = oracle.paged_logits(w.q, w.kv_fused, w.weights, w.block_tables,
                                           w.seq_lens, w.max_seq_len, block_size=w.block_size)
            kth = torch.from_numpy(kth_values(ref, expected_row_ends(w), w.top_k))
            thr0 = synth.thresholds_scaled_kth(w, kth)
        thr.copy_(thr0.to(d))
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert (row_ends.cpu().numpy() == expected_row_ends(w)).all()
        check_logits(w, out, ref, tol, untouched_fill_nan=False)
        res = {"thresholds": thr.cpu().numpy(), "counters": counters.cpu().numpy(),
               "candidates": cand.cpu().numpy(), "arrivals": arrivals.cpu().numpy(),
               "ranges": ranges.cpu().numpy()}
        check_selection(out.cpu().numpy(), expected_row_ends(w), w.top_k, w.capacity, res,
                        thr0.numpy())
        # Eager run on the same inputs gives bit-identical logits and the same selection.
        graph_logits = out.clone()
        def selection():
            c, rg, lc = cand.cpu().numpy(), ranges.cpu().numpy(), out.cpu().numpy()
            k = np.minimum(expected_row_ends(w), w.top_k)
            return [selected_from_slots(lc[r], c[r], rg[0, r], rg[1, r], int(k[r])).tolist()
                    for r in range(rows)]
        graph_sel = selection()
        thr.copy_(thr0.to(d))
        with torch.cuda.stream(s):
            step()
        torch.cuda.synchronize()
        assert torch.equal(out, graph_logits)
        assert graph_sel == selection()
    assert idx.device_status(clear=True) == 0
