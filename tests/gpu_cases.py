"""Helpers shared by the GPU parity tests: move a seeded workload to the device, run the CUDA
path through the C ABI, and compare with the CPU oracle."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import paged_fp8_mqa_gb300 as idx
from paged_fp8_mqa_gb300 import synth

# Logits tolerance: |gpu - oracle| <= REL * |scale| * sum_h |w_h relu(s_h)| + ABS.
REL = 2e-6
ABS = 1e-7


def dev():
    return torch.device("cuda:0")


def to_device(w: synth.Workload):
    d = dev()
    return dict(q=w.q.to(d), kv=w.kv_fused.to(d), weights=w.weights.to(d),
                bt=w.block_tables.to(d), seq_lens=w.seq_lens.to(d))


def gpu_logits(w: synth.Workload, *, schedule=False, num_sms=0, fill=float("nan"), tensors=None,
               bt=None, seq_lens=None):
    t = tensors or to_device(w)
    pad = idx.idx_padded_seq_len(w.max_seq_len)
    out = torch.full((w.rows, pad), fill, dtype=torch.float32, device=dev())
    row_ends = torch.full((w.rows,), -7, dtype=torch.int32, device=dev())
    sl = t["seq_lens"] if seq_lens is None else seq_lens
    sched = idx.schedule(sl, w.next_n, num_sms) if schedule else None
    idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"] if bt is None else bt, sl,
                   w.max_seq_len, out=out, schedule_meta=sched, num_sms=num_sms,
                   row_ends_out=row_ends)
    torch.cuda.synchronize()
    return out, row_ends


@functools.lru_cache(maxsize=8)
def oracle_logits_cached(name: str):
    w = synth.WORKLOADS[name]()
    ref, tol = oracle.paged_logits(w.q, w.kv_fused, w.weights, w.block_tables, w.seq_lens,
                                   w.max_seq_len, block_size=w.block_size)
    return w, ref, tol


def check_logits(w: synth.Workload, got_t: torch.Tensor, ref: np.ndarray, tol: np.ndarray,
                 untouched_fill_nan: bool = True) -> dict:
    """Element-wise check of every in-extent score; zero-length requests' rows untouched;
    columns at or past seq_lens[b] untouched (this build writes only p < seq_lens[b])."""
    got = got_t.cpu().double().numpy()
    re = w.row_ends().numpy()
    worst = 0.0
    n_checked = 0
    for r in range(w.rows):
        L = int(w.seq_lens[r // w.next_n])
        e = int(re[r])
        if e:
            err = np.abs(got[r, :e] - ref[r, :e])
            lim = REL * tol[r, :e] + ABS
            bad = np.nonzero(~(err <= lim))[0]
            assert bad.size == 0, (
                f"row {r}: {bad.size} scores out of tolerance, first p={bad[0]} "
                f"gpu={got[r, bad[0]]} oracle={ref[r, bad[0]]} tol={lim[bad[0]]}")
            worst = max(worst, float(np.max(err / (tol[r, :e] + 1e-30))))
            n_checked += e
        if untouched_fill_nan:
            assert np.isnan(got[r, L:]).all(), f"row {r}: columns >= seq_len were written"
    return {"checked": n_checked, "worst_rel": worst}
