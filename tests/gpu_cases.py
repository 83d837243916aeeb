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


def expected_row_ends(w: synth.Workload) -> np.ndarray:
    """int32 [rows]: the oracle's extent of every row (row b*next_n + t sees positions
    0 .. seq_lens[b] - next_n + t).  Every GPU test takes its expected extents from here."""
    return oracle.row_ends(w.seq_lens, w.next_n)


def expected_scores(w: synth.Workload) -> int:
    """Number of (row, position) pairs inside the oracle's extents."""
    return int(expected_row_ends(w).astype(np.int64).sum())


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
    re = expected_row_ends(w)
    worst = 0.0
    n_checked = 0
    for r in range(w.rows):
        L = int(w.seq_lens[r // w.next_n])
        e = int(re[r])
        # The oracle leaves exactly the columns outside the row's extent unset (NaN).
        assert np.isfinite(ref[r, :e]).all() and np.isnan(ref[r, e:]).all(), \
            f"row {r}: the oracle's logits disagree with its own extent {e}"
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


# ---- threshold select ----------------------------------------------------------------------

def order_keys(x: np.ndarray) -> np.ndarray:
    """uint32 keys whose unsigned order is IEEE totalOrder of the float32 values."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return np.where(u >> 31 == 1, ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def kth_values(ref: np.ndarray, row_ends: np.ndarray, top_k: int) -> np.ndarray:
    """Each row's K'-th largest value of a float64 logits array (NaN for empty rows)."""
    out = np.full(len(row_ends), np.nan)
    for r, e in enumerate(row_ends):
        k = min(int(e), top_k)
        if k:
            out[r] = np.partition(ref[r, :e], e - k)[e - k]
    return out


def gpu_select(logits: torch.Tensor, row_ends: torch.Tensor, thresholds: torch.Tensor,
               top_k: int, capacity: int, max_context: int, repair: bool = True):
    rows = row_ends.shape[0]
    d = logits.device
    thr = thresholds.clone().to(d)
    counters = torch.zeros(rows, 2, dtype=torch.int32, device=d)
    cand = torch.full((rows, top_k + capacity, 2), -1, dtype=torch.int32, device=d)
    arrivals = torch.zeros(rows, dtype=torch.int32, device=d) if repair else None
    ranges = torch.full((2, rows), -1, dtype=torch.int32, device=d) if repair else None
    idx.threshold_select(logits, row_ends, thr, counters, cand, top_k, capacity, max_context,
                         arrivals=arrivals, ranges=ranges)
    torch.cuda.synchronize()
    res = dict(thresholds=thr.cpu().numpy(), counters=counters.cpu().numpy(),
               candidates=cand.cpu().numpy())
    if repair:
        res["arrivals"] = arrivals.cpu().numpy()
        res["ranges"] = ranges.cpu().numpy()
    return res


def selected_from_slots(logits_row: np.ndarray, cand_row: np.ndarray, lo: int, hi: int,
                        k: int) -> np.ndarray:
    """The row's top-k as the slots [lo, hi) give it: order the stored (index, bits) pairs by
    totalOrder of the stored bits, descending, then index ascending, and take k."""
    items = cand_row[lo:hi]
    idxs = items[:, 0].astype(np.int64)
    bits = items[:, 1].astype(np.int32).view(np.float32)
    assert len(np.unique(idxs)) == len(idxs), "a key is stored twice"
    assert (bits.view(np.uint32) == logits_row[idxs].view(np.uint32)).all(), \
        "stored score bits differ from the logits"
    order = np.lexsort((idxs, ~order_keys(bits)))
    return idxs[order][:k]


def check_selection(logits_cpu: np.ndarray, row_ends: np.ndarray, top_k: int, capacity: int,
                    res: dict, thr_in: np.ndarray):
    """Every row holds exactly its top-K' (ties to the lowest index) in [ranges[0], ranges[1]);
    rows that fit their input threshold keep true counts; repaired rows get their K'-th value as
    threshold and exactly K' items; arrivals are back to zero."""
    top, cnt = oracle.topk(logits_cpu, row_ends, top_k)
    nc, nt, fits = oracle.select_classify(logits_cpu, row_ends, thr_in, top_k, capacity)
    rg = res["ranges"]
    repaired = 0
    for r in range(len(row_ends)):
        k = int(cnt[r])
        got = selected_from_slots(logits_cpu[r], res["candidates"][r], rg[0, r], rg[1, r], k)
        assert (got == top[r, :k]).all(), f"row {r}: selection differs from the exact top-k"
        if fits[r]:
            assert tuple(res["counters"][r]) == (nc[r], nt[r]), f"row {r} counters"
            assert rg[0, r] == top_k - min(nt[r], top_k) and rg[1, r] == top_k + min(nc[r], capacity)
            assert np.float32(res["thresholds"][r]).tobytes() == np.float32(thr_in[r]).tobytes()
        else:
            repaired += 1
            c, m = res["counters"][r]
            assert c + m == k and rg[1, r] - rg[0, r] == k, f"row {r}: repaired counts"
            kth = logits_cpu[r, top[r, k - 1]]
            assert np.float32(res["thresholds"][r]).tobytes() == np.float32(kth).tobytes(), \
                f"row {r}: repaired threshold is not the K'-th value"
    assert (res["arrivals"] == 0).all(), "arrivals not returned to zero"
    return repaired
