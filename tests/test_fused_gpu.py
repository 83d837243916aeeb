"""Fused score + threshold select (no logits written) against the two-stage path on the same
inputs: the logits kernel's float32 scores, then the select kernel.  Both compute each score by
the same arithmetic, so every output must agree exactly (slots compared as sets); the selection
itself is checked against the oracle's exact top-k of those scores."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_fp8_mqa_gb300 as idx
from paged_fp8_mqa_gb300 import synth
from gpu_cases import (expected_row_ends, expected_scores, check_selection, gpu_logits, gpu_select, kth_values, selected_from_slots,
                       to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    idx.device_status(clear=True)
    yield
    assert idx.device_status(clear=True) == 0, "a kernel raised a device status bit"


def gpu_fused(w, t, thresholds, top_k, capacity, repair=True, num_sms=0):
    d = t["q"].device
    rows = w.rows
    thr = thresholds.clone().to(d)
    counters = torch.zeros(rows, 2, dtype=torch.int32, device=d)
    cand = torch.full((rows, top_k + capacity, 2), -1, dtype=torch.int32, device=d)
    arrivals = torch.zeros(w.batch, dtype=torch.int32, device=d) if repair else None
    ranges = torch.full((2, rows), -1, dtype=torch.int32, device=d) if repair else None
    idx.indexer_threshold_select(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"],
                                 w.max_seq_len, thresholds=thr, counters=counters,
                                 candidates=cand, top_k=top_k, arrivals=arrivals, ranges=ranges,
                                 num_sms=num_sms)
    torch.cuda.synchronize()
    res = dict(thresholds=thr.cpu().numpy(), counters=counters.cpu().numpy(),
               candidates=cand.cpu().numpy())
    if repair:
        res["arrivals"] = arrivals.cpu().numpy()
        res["ranges"] = ranges.cpu().numpy()
    return res


def slot_sets(res, r, top_k):
    lo, hi = res["ranges"][0, r], res["ranges"][1, r]
    return {tuple(x) for x in res["candidates"][r, lo:hi].tolist()}


def compare(w, logits, thr, top_k, capacity, num_sms=0, t=None):
    """Fused vs two-stage on the same thresholds; returns the number of repaired rows."""
    t = t or to_device(w)
    lc = logits.cpu().numpy()
    re = expected_row_ends(w)
    row_ends = torch.from_numpy(re).to(torch.int32).cuda()
    two = gpu_select(logits, row_ends, thr, top_k, capacity, w.max_seq_len)
    fused = gpu_fused(w, t, thr, top_k, capacity, num_sms=num_sms)
    repaired = check_selection(lc, re, top_k, capacity, fused, thr.numpy())
    assert (fused["counters"] == two["counters"]).all(), "counters differ from the two-stage path"
    assert (fused["ranges"] == two["ranges"]).all(), "ranges differ from the two-stage path"
    assert fused["thresholds"].tobytes() == two["thresholds"].tobytes(), "thresholds differ"
    for r in range(w.rows):
        assert slot_sets(fused, r, top_k) == slot_sets(two, r, top_k), f"row {r}: slots differ"
    return repaired


def _small(seed, next_n, lens, block_size=64, max_seq_len=None, num_heads=64, head_dim=128):
    m = max_seq_len or max(max(lens), 1)
    return synth.make_workload("edge", seed, len(lens), next_n, m, "fixed", values=list(lens),
                               block_size=block_size, num_heads=num_heads, head_dim=head_dim)


def _threshold_variants(lc, re, top_k, seed):
    kth = kth_values(lc.astype(np.float64), re, top_k)
    base = torch.from_numpy(np.nan_to_num(kth, nan=0.0)).to(torch.float32)
    g = torch.Generator().manual_seed(seed)
    mixed = base.clone()
    pick = torch.randperm(len(base), generator=g)
    mixed[pick[0::4]] = math.inf
    mixed[pick[1::4]] = -math.inf
    mixed[pick[2::4]] = math.nan
    return {"kth": base, "below": base - 0.05 * base.abs() - 1e-3, "mixed": mixed,
            "inf": torch.full_like(base, math.inf), "nan": torch.full_like(base, math.nan)}


CASES = [
    (1, 64, [5000, 1, 0, 777, 4096, 129]),
    (2, 64, [3000, 0, 2, 64, 65, 9000]),
    (3, 32, [2500, 3, 2, 0, 1300, 6000, 31, 33]),
    (4, 128, [4000, 4, 3, 100, 0, 8191, 8193]),
    (4, 64, [12000, 700, 5, 1, 20000]),
]


@pytest.mark.parametrize("next_n,block_size,lens", CASES,
                         ids=[f"n{n}-bs{b}-{len(l)}req" for n, b, l in CASES])
@pytest.mark.parametrize("top_k,capacity", [(64, 63), (256, 1000)])
def test_fused_matches_two_stage(next_n, block_size, lens, top_k, capacity):
    w = _small(500 + next_n + block_size, next_n, lens, block_size=block_size)
    t = to_device(w)
    logits, _ = gpu_logits(w, fill=0.0, tensors=t)
    lc = logits.cpu().numpy()
    re = expected_row_ends(w)
    for name, thr in _threshold_variants(lc, re, top_k, seed=next_n).items():
        repaired = compare(w, logits, thr, top_k, capacity, t=t)
        if name == "inf":
            assert repaired == int((re > 0).sum())


@pytest.mark.parametrize("name", ["serving", "long_select"])
def test_fused_full_workloads(name):
    w = synth.WORKLOADS[name]()
    t = to_device(w)
    logits, _ = gpu_logits(w, fill=0.0, tensors=t)
    re = expected_row_ends(w)
    kth = torch.from_numpy(kth_values(logits.cpu().double().numpy(), re, w.top_k))
    thr = (synth.thresholds_below_kth(w, kth) if name == "long_select"
           else synth.thresholds_scaled_kth(w, kth))
    repaired = compare(w, logits, thr, w.top_k, w.capacity, t=t)
    if name == "long_select":
        assert repaired >= 10


@pytest.mark.parametrize("num_sms", [1, 3])
def test_fused_runs_over_several_tile_lists(num_sms):
    """Few CTAs: each run spans several tile lists and many requests, so a request's rows are
    classified by warps of several lists (and CTAs), and the rescoring launch's own work split
    covers the requests left to repair."""
    g = torch.Generator().manual_seed(77)
    lens = torch.randint(1, 700, (160,), generator=g).tolist()
    lens[5:9] = [0, 1, 2, 3]
    w = _small(520 + num_sms, 2, lens)
    t = to_device(w)
    logits, _ = gpu_logits(w, fill=0.0, tensors=t)
    lc = logits.cpu().numpy()
    variants = _threshold_variants(lc, expected_row_ends(w), 32, seed=num_sms)
    for thr in (variants["kth"], variants["mixed"]):
        compare(w, logits, thr, 32, 40, num_sms=num_sms, t=t)


def test_fused_without_arrivals_counts_only():
    """No arrivals: one launch, true counts, and stored slots holding valid (index, bits) pairs
    of the right kind; nothing is repaired."""
    w = _small(530, 3, [3000, 40, 0, 2, 5000])
    t = to_device(w)
    logits, _ = gpu_logits(w, fill=0.0, tensors=t)
    lc = logits.cpu().numpy()
    re = expected_row_ends(w)
    top_k, capacity = 128, 200
    for thr in _threshold_variants(lc, re, top_k, seed=9).values():
        res = gpu_fused(w, t, thr, top_k, capacity, repair=False)
        nc, nt, _ = oracle.select_classify(lc, re, thr.numpy(), top_k, capacity)
        assert (res["counters"][:, 0] == nc).all() and (res["counters"][:, 1] == nt).all()
        assert res["thresholds"].tobytes() == thr.numpy().tobytes()
        for r in range(w.rows):
            c = res["candidates"][r]
            for items, is_c in ((c[top_k:top_k + min(nc[r], capacity)], True),
                                (c[top_k - min(nt[r], top_k):top_k], False)):
                if len(items) == 0:
                    continue
                i = items[:, 0]
                assert len(np.unique(i)) == len(i) and (i >= 0).all() and (i < re[r]).all()
                v = lc[r, i]
                assert (items[:, 1].astype(np.int32).view(np.float32).view(np.uint32)
                        == v.view(np.uint32)).all()
                tr = thr.numpy()[r]
                assert (v > tr).all() if is_c else (~(v > tr) & ~(v < tr)).all()


def test_fused_graph_replay_and_repeat():
    """Captured once and replayed: the same selection as eager calls, arrivals back at zero
    after every call, the repair launches included."""
    w = _small(540, 2, [9000, 300, 0, 4000, 77])
    t = to_device(w)
    logits, _ = gpu_logits(w, fill=0.0, tensors=t)
    lc = logits.cpu().numpy()
    re = expected_row_ends(w)
    top_k, capacity = 100, 120
    thr0 = _threshold_variants(lc, re, top_k, seed=4)["mixed"].cuda()
    d = t["q"].device
    thr = thr0.clone()
    counters = torch.zeros(w.rows, 2, dtype=torch.int32, device=d)
    cand = torch.zeros(w.rows, top_k + capacity, 2, dtype=torch.int32, device=d)
    arrivals = torch.zeros(w.batch, dtype=torch.int32, device=d)
    ranges = torch.zeros(2, w.rows, dtype=torch.int32, device=d)
    scratch = torch.empty(w.rows, idx.idx_padded_seq_len(w.max_seq_len), device=d)

    def step():
        counters.zero_()
        thr.copy_(thr0)
        idx.indexer_threshold_select(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"],
                                     w.max_seq_len, thresholds=thr, counters=counters,
                                     candidates=cand, top_k=top_k, arrivals=arrivals,
                                     ranges=ranges, scratch=scratch)

    def selection():
        c, rg = cand.cpu().numpy(), ranges.cpu().numpy()
        k = np.minimum(re, top_k)
        return [selected_from_slots(lc[r], c[r], rg[0, r], rg[1, r], int(k[r])).tolist()
                for r in range(w.rows)]

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    first = selection()
    assert (arrivals == 0).all()
    top, cnt = oracle.topk(lc, re, top_k)
    for r in range(w.rows):
        assert first[r] == top[r, :cnt[r]].tolist()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for _ in range(2):
        cand.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert (arrivals == 0).all()
        assert selection() == first


@pytest.mark.parametrize("next_n", [1, 4])
def test_fused_empty_and_short_requests(next_n):
    """Requests with no keys at all, or fewer than next_n (some rows empty): every row fits
    with nothing stored (K' = 0) or holds its few keys; ranges are written for all rows."""
    for lens in ([0, 0, 0], [0, 1, 0, 2, 3]):
        w = _small(560 + next_n + len(lens), next_n, lens, max_seq_len=256)
        t = to_device(w)
        logits, _ = gpu_logits(w, fill=0.0, tensors=t)
        thr = torch.full((w.rows,), math.inf)
        compare(w, logits, thr, 16, 15, t=t)
        fused = gpu_fused(w, t, thr, 16, 15)
        re = expected_row_ends(w)
        for r in range(w.rows):
            assert fused["ranges"][1, r] - fused["ranges"][0, r] == min(int(re[r]), 16)


@pytest.mark.parametrize("next_n", [1, 2, 4])
def test_fused_32_heads(next_n):
    w = _small(570 + next_n, next_n, [4000, 3, 0, 900, 7000], num_heads=32)
    t = to_device(w)
    logits, _ = gpu_logits(w, fill=0.0, tensors=t)
    lc = logits.cpu().numpy()
    for thr in _threshold_variants(lc, expected_row_ends(w), 64, seed=next_n).values():
        compare(w, logits, thr, 64, 63, t=t)


@pytest.mark.parametrize("next_n,heads", [(1, 64), (4, 64), (2, 32)])
def test_fused_head_dim_64(next_n, heads):
    w = _small(580 + next_n + heads, next_n, [4000, 3, 0, 900, 7000], num_heads=heads,
               head_dim=64)
    t = to_device(w)
    logits, _ = gpu_logits(w, fill=0.0, tensors=t)
    lc = logits.cpu().numpy()
    for thr in _threshold_variants(lc, expected_row_ends(w), 64, seed=next_n).values():
        compare(w, logits, thr, 64, 63, t=t)
