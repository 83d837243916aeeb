"""Threshold top-k select: the CUDA path against the oracle's top-k on the GPU's own logits."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_fp8_mqa_gb300 as idx
from paged_fp8_mqa_gb300 import synth
from gpu_cases import (expected_row_ends, expected_scores, check_selection, gpu_logits, gpu_select, kth_values, oracle_logits_cached,
                       selected_from_slots)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    idx.device_status(clear=True)
    yield
    assert idx.device_status(clear=True) == 0, "a kernel raised a device status bit"


def _logits_and_thresholds(name):
    w, ref, _ = oracle_logits_cached(name)
    got, row_ends = gpu_logits(w, fill=0.0)
    re = expected_row_ends(w)
    kth = torch.from_numpy(kth_values(ref, re, w.top_k))
    if name == "long_select":
        thr = synth.thresholds_below_kth(w, kth)
    else:
        thr = synth.thresholds_scaled_kth(w, kth)
    return w, got, row_ends, thr


@pytest.mark.parametrize("name", ["long_select", "serving"])
def test_full_workload_selection(name):
    w, logits, row_ends, thr = _logits_and_thresholds(name)
    res = gpu_select(logits, row_ends, thr.cuda(), w.top_k, w.capacity, w.max_seq_len)
    lc = logits.cpu().numpy()
    repaired = check_selection(lc, expected_row_ends(w), w.top_k, w.capacity, res, thr.numpy())
    if name == "long_select":
        assert repaired >= 10  # the ten rows forced to +inf at least


def test_any_threshold_gives_the_same_selection():
    w, logits, row_ends, thr = _logits_and_thresholds("long_select")
    lc = logits.cpu().numpy()
    re = expected_row_ends(w)
    sets = []
    g = torch.Generator().manual_seed(5)
    variants = [thr, torch.full_like(thr, math.inf), torch.full_like(thr, -math.inf),
                torch.full_like(thr, math.nan), thr + torch.randn(thr.shape, generator=g)]
    for t in variants:
        res = gpu_select(logits, row_ends, t.cuda(), w.top_k, w.capacity, w.max_seq_len)
        check_selection(lc, re, w.top_k, w.capacity, res, t.numpy())
        k = np.minimum(re, w.top_k)
        sets.append([selected_from_slots(lc[r], res["candidates"][r], res["ranges"][0, r],
                                         res["ranges"][1, r], int(k[r])).tolist()
                     for r in range(len(re))])
    for s in sets[1:]:
        assert s == sets[0]


def _synthetic(rows, n, kind, seed=0):
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        x = torch.randn(rows, n, generator=g)
    elif kind == "ties":
        x = torch.randint(-3, 4, (rows, n), generator=g).to(torch.float32)
    elif kind == "constant":
        x = torch.full((rows, n), 0.5)
    elif kind == "zeros":
        x = torch.zeros(rows, n)
        x[:, ::3] = -0.0
    return x


@pytest.mark.parametrize("kind", ["normal", "ties", "constant", "zeros"])
@pytest.mark.parametrize("top_k,capacity", [(64, 63), (64, 200), (1, 0), (300, 299)])
def test_small_rows(kind, top_k, capacity):
    rows, n = 9, 20000
    x = _synthetic(rows, n, kind, seed=top_k)
    row_ends = torch.tensor([n, 0, 1, 63, 64, 65, 8191, 8193, 19999], dtype=torch.int32)
    stride = 20480
    logits = torch.zeros(rows, stride)
    logits[:, :n] = x
    lc = logits.numpy()
    kth = kth_values(lc.astype(np.float64), row_ends.numpy(), top_k)
    thr = torch.from_numpy(np.nan_to_num(kth, nan=0.0)).to(torch.float32)
    for t in (thr, thr - 0.25, torch.full_like(thr, math.inf)):
        res = gpu_select(logits.cuda(), row_ends.cuda(), t.cuda(), top_k, capacity, n)
        check_selection(lc, row_ends.numpy(), top_k, capacity, res, t.numpy())


def test_nan_and_equal_scores_are_ties():
    """Classification alone (no repair): s > thr is a candidate, s == thr or NaN a tie."""
    n = 1000
    x = torch.randn(2, n, generator=torch.Generator().manual_seed(3))
    x[0, 10] = math.nan
    x[0, 20] = 0.25
    x[0, 30] = 0.25
    x[1, :] = 0.25
    thr = torch.tensor([0.25, 0.25])
    row_ends = torch.tensor([n, n], dtype=torch.int32)
    res = gpu_select(x.cuda(), row_ends.cuda(), thr.cuda(), 64, 2000, n, repair=False)
    nc, nt, _ = oracle.select_classify(x, row_ends, thr, 64, 2000)
    assert (res["counters"][:, 0] == nc).all() and (res["counters"][:, 1] == nt).all()
    tie_idx = sorted(res["candidates"][0, 64 - nt[0]:64, 0])
    assert tie_idx == [10, 20, 30]


def test_classification_only_slots():
    """Without arrivals: true counts, and the first capacity candidates / top_k ties stored
    at the slot positions the select's Parameters give, each holding its key and score bits."""
    w, logits, row_ends, thr = _logits_and_thresholds("serving")
    lc = logits.cpu().numpy()
    re = expected_row_ends(w)
    res = gpu_select(logits, row_ends, thr.cuda(), w.top_k, w.capacity, w.max_seq_len,
                     repair=False)
    nc, nt, _ = oracle.select_classify(lc, re, thr.numpy(), w.top_k, w.capacity)
    assert (res["counters"][:, 0] == nc).all() and (res["counters"][:, 1] == nt).all()
    for r in range(len(re)):
        tk = w.top_k
        c = res["candidates"][r]
        stored_c = c[tk:tk + min(nc[r], w.capacity)]
        stored_t = c[tk - min(nt[r], tk):tk]
        for items, is_c in ((stored_c, True), (stored_t, False)):
            if len(items) == 0:
                continue
            i = items[:, 0]
            assert len(np.unique(i)) == len(i) and (i >= 0).all() and (i < re[r]).all()
            v = lc[r, i]
            assert (items[:, 1].astype(np.int32).view(np.float32).view(np.uint32)
                    == v.view(np.uint32)).all()
            t = thr.numpy()[r]
            assert (v > t).all() if is_c else (~(v > t) & ~(v < t)).all()


def test_arrivals_stay_zero_across_calls():
    w, logits, row_ends, thr = _logits_and_thresholds("long_select")
    d = logits.device
    rows = row_ends.shape[0]
    arrivals = torch.zeros(rows, dtype=torch.int32, device=d)
    ranges = torch.zeros(2, rows, dtype=torch.int32, device=d)
    cand = torch.zeros(rows, w.top_k + w.capacity, 2, dtype=torch.int32, device=d)
    first = None
    for it in range(3):
        counters = torch.zeros(rows, 2, dtype=torch.int32, device=d)
        t = thr.cuda()
        idx.threshold_select(logits, row_ends, t, counters, cand, w.top_k, w.capacity,
                             w.max_seq_len, arrivals=arrivals, ranges=ranges)
        torch.cuda.synchronize()
        assert (arrivals == 0).all()
        c = cand.cpu().numpy()
        rg = ranges.cpu().numpy()
        lc = logits.cpu().numpy()
        k = np.minimum(expected_row_ends(w), w.top_k)
        sel = [selected_from_slots(lc[r], c[r], rg[0, r], rg[1, r], int(k[r])).tolist()
               for r in range(rows)]
        first = first or sel
        assert sel == first


@pytest.mark.parametrize("kind", ["normal", "ties"])
def test_very_long_rows(kind):
    """Rows of up to 270000 keys (33 classifying CTAs each), each repaired by one CTA of the
    finishing launch."""
    rows, n = 3, 270000
    x = _synthetic(rows, n, kind, seed=9)
    row_ends = torch.tensor([n, 262145, 70000], dtype=torch.int32)
    lc = x.numpy()
    top_k, capacity = 2048, 4096
    kth = kth_values(lc.astype(np.float64), row_ends.numpy(), top_k)
    thr = torch.from_numpy(np.nan_to_num(kth, nan=0.0)).to(torch.float32)
    for t in (thr, torch.full_like(thr, math.inf), thr - 1.0):
        res = gpu_select(x.cuda(), row_ends.cuda(), t.cuda(), top_k, capacity, n)
        check_selection(lc, row_ends.numpy(), top_k, capacity, res, t.numpy())


@pytest.mark.parametrize("max_context", [32768, 100000, 262144])
def test_row_lengths_around_chunks(max_context):
    """Rows spread over 4 to 32 classifying CTAs, with ragged ends around the chunks' borders,
    thresholds that fit and that force the repair, and a row of many equal keys (the bin of the
    K'-th value too full for the repair's shared-memory buffer)."""
    g = torch.Generator().manual_seed(max_context)
    ends = [max_context, max_context - 1, 32767, 32769, 65537, 5000, 1, 0]
    ends = [min(e, max_context) for e in ends]
    rows = len(ends)
    x = torch.randn(rows, max_context, generator=g)
    x[1, :] = torch.randint(-2, 3, (max_context,), generator=g).to(torch.float32)  # many ties
    lc = x.numpy()
    row_ends = torch.tensor(ends, dtype=torch.int32)
    for top_k, capacity in ((2048, 4096), (300, 299)):
        kth = kth_values(lc.astype(np.float64), row_ends.numpy(), top_k)
        thr = torch.from_numpy(np.nan_to_num(kth, nan=0.0)).to(torch.float32)
        for t in (thr, torch.full_like(thr, math.inf), thr - 0.5):
            res = gpu_select(x.cuda(), row_ends.cuda(), t.cuda(), top_k, capacity, max_context)
            check_selection(lc, row_ends.numpy(), top_k, capacity, res, t.numpy())


@pytest.mark.parametrize("top_k,capacity", [(300, 299), (2048, 4096)])
def test_repair_with_nan_inf_and_signed_zeros(top_k, capacity):
    """Repairs (rows longer than the repair's buffer, and rows of at most top_k keys) over keys
    that include +NaN and -NaN (above +inf and below -inf in totalOrder), +-inf and +-0.  The
    thresholds +inf and -inf make every long row need a repair (no candidates, or all of them);
    a threshold that lets such a row fit would count its NaNs as ties, which the fit rule treats
    as the threshold's value rather than by totalOrder, so only repaired rows are compared."""
    g = torch.Generator().manual_seed(77 + top_k)
    rows, n = 6, 20000
    x = torch.randn(rows, n, generator=g).abs()  # non-negative: the gathering bound is >= +0
    x[1] = 0.0
    x[1, ::2] = -0.0
    nan_pos = np.frombuffer(np.array([0x7FC00001], dtype=np.uint32).tobytes(), dtype=np.float32)[0]
    nan_neg = np.frombuffer(np.array([0xFFC00002], dtype=np.uint32).tobytes(), dtype=np.float32)[0]
    for r in range(rows):
        idx_ = torch.randperm(n, generator=g)[:40]
        x[r, idx_[:10]] = float(nan_pos)
        x[r, idx_[10:20]] = float(nan_neg)
        x[r, idx_[20:30]] = math.inf
        x[r, idx_[30:40]] = -math.inf
    lc = x.numpy()
    row_ends = torch.tensor([n, n, 15000, top_k, max(top_k - 7, 1), 9000], dtype=torch.int32)
    for t in (torch.full((rows,), math.inf), torch.full((rows,), -math.inf)):
        res = gpu_select(x.cuda(), row_ends.cuda(), t.cuda(), top_k, capacity, n)
        check_selection(lc, row_ends.numpy(), top_k, capacity, res, t.numpy())


def test_many_rows_per_finishing_cta():
    """More rows than SMs: each CTA of the finishing launch applies the fit rule to several rows
    and repairs several rows one after another.  Lengths from 0 to 20000, thresholds that fit,
    that force a repair (+inf) and that are a little low (too many candidates for capacity =
    top_k - 1); arrivals holds garbage on entry (it is only the switch) and is zero after."""
    g = torch.Generator().manual_seed(404)
    rows, n = 400, 20000
    x = torch.randn(rows, n, generator=g)
    x[7] = torch.randint(-2, 3, (n,), generator=g).to(torch.float32)  # many ties
    ends = torch.randint(0, n + 1, (rows,), generator=g)
    ends[:4] = torch.tensor([0, 1, n, 64])
    row_ends = ends.to(torch.int32)
    lc = x.numpy()
    top_k, capacity = 64, 63
    kth = kth_values(lc.astype(np.float64), row_ends.numpy(), top_k)
    kth = torch.from_numpy(np.nan_to_num(kth, nan=0.0)).to(torch.float32)
    kind = torch.arange(rows) % 3
    thr = torch.where(kind == 0, kth, torch.where(kind == 1, torch.full_like(kth, math.inf),
                                                   kth - 0.25))
    d = torch.device("cuda")
    t = thr.clone().to(d)
    counters = torch.zeros(rows, 2, dtype=torch.int32, device=d)
    cand = torch.full((rows, top_k + capacity, 2), -1, dtype=torch.int32, device=d)
    arrivals = torch.full((rows,), 7, dtype=torch.int32, device=d)
    ranges = torch.full((2, rows), -1, dtype=torch.int32, device=d)
    idx.threshold_select(x.to(d), row_ends.to(d), t, counters, cand, top_k, capacity, n,
                         arrivals=arrivals, ranges=ranges)
    torch.cuda.synchronize()
    res = dict(thresholds=t.cpu().numpy(), counters=counters.cpu().numpy(),
               candidates=cand.cpu().numpy(), arrivals=arrivals.cpu().numpy(),
               ranges=ranges.cpu().numpy())
    repaired = check_selection(lc, row_ends.numpy(), top_k, capacity, res, thr.numpy())
    assert repaired >= rows // 3 - 10  # the +inf rows with at least one key, and more


def test_thousands_of_short_rows():
    """2500 short rows of 0..3000 keys (16 rows per finishing CTA); thresholds that fit and +inf
    (a repair for every non-empty row)."""
    g = torch.Generator().manual_seed(2500)
    rows, n = 2500, 3000
    x = torch.randn(rows, n, generator=g)
    row_ends = torch.randint(0, n + 1, (rows,), generator=g).to(torch.int32)
    row_ends[:3] = torch.tensor([0, n, 1], dtype=torch.int32)
    stride = 3072
    logits = torch.zeros(rows, stride)
    logits[:, :n] = x
    lc = logits.numpy()
    top_k, capacity = 32, 31
    kth = kth_values(lc.astype(np.float64), row_ends.numpy(), top_k)
    kth = torch.from_numpy(np.nan_to_num(kth, nan=0.0)).to(torch.float32)
    thr = torch.where(torch.arange(rows) % 2 == 0, kth, torch.full_like(kth, math.inf))
    res = gpu_select(logits.cuda(), row_ends.cuda(), thr.cuda(), top_k, capacity, n)
    repaired = check_selection(lc, row_ends.numpy(), top_k, capacity, res, thr.numpy())
    assert repaired >= rows // 2 - 10
