"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``check_*`` takes a loaded oracle library (the real build, or a deliberately broken one in
the mutation test) and raises AssertionError when the oracle disagrees with:
  * values the pages print (tests/golden/worked_examples.json, each entry cited there);
  * library routines on special cases (torch's float8 decode, float64 matmul, torch.topk,
    numpy.lexsort);
  * closed forms and invariants that hold for the indexer's definition.
"""
from __future__ import annotations

import json
import math
import os
import struct

import numpy as np
import torch

import oracle
from paged_fp8_mqa_gb300 import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "worked_examples.json")))


# --------------------------------------------------------------------------------------------
# Independent references built from library routines
# --------------------------------------------------------------------------------------------

def dense_reference(w: synth.Workload) -> np.ndarray:
    """Logits via torch float64 matmul on each request's de-paged K (values and scales sliced
    out of kv_fused with tensor views), NaN outside the extents."""
    bs, D = w.block_size, w.head_dim
    vals = (w.kv_fused[:, :bs * D].contiguous().view(torch.float8_e4m3fn)
            .view(-1, bs, D).to(torch.float64))
    scl = w.kv_fused[:, bs * D:].contiguous().view(torch.float32).view(-1, bs).to(torch.float64)
    q = w.q.view(torch.float8_e4m3fn).to(torch.float64)
    wt = w.weights.to(torch.float64)
    n = w.next_n
    out = torch.full((w.rows, oracle.padded_seq_len(w.max_seq_len)), float("nan"),
                     dtype=torch.float64)
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        if L == 0:
            continue
        pages = w.block_tables[b, :math.ceil(L / bs)].long()
        K = vals[pages].reshape(-1, D)[:L]
        S = scl[pages].reshape(-1)[:L]
        for t in range(n):
            re = L - n + t + 1
            if re <= 0:
                continue
            scores = q[b, t] @ K[:re].T                      # [H, re]
            out[b * n + t, :re] = S[:re] * (wt[b * n + t] @ scores.clamp_min(0))
    return out.numpy()


def _small(seed=11, batch=3, next_n=3, lens=(70, 5, 129), max_seq_len=160, block_size=32,
           heads=8, head_dim=32, **kw) -> synth.Workload:
    return synth.make_workload("pin", seed, batch, next_n, max_seq_len, "fixed",
                               values=list(lens), num_heads=heads, head_dim=head_dim,
                               block_size=block_size, **kw)


def _logits(lib, w: synth.Workload, **kw):
    return oracle.paged_logits(w.q, w.kv_fused, w.weights, w.block_tables, w.seq_lens,
                               w.max_seq_len, block_size=w.block_size, lib=lib, **kw)


def _same(a, b, rtol=1e-12, scale=None):
    """NaN in the same places, values equal to rtol (relative to ``scale`` when given)."""
    na, nb = np.isnan(a), np.isnan(b)
    assert (na == nb).all(), f"NaN pattern differs at {np.argwhere(na != nb)[:5].tolist()}"
    m = ~na
    ref = np.abs(b[m]) if scale is None else scale[m]
    err = np.abs(a[m] - b[m])
    assert (err <= rtol * ref + 1e-300).all(), f"max err {err.max()} (ref {ref[err.argmax()]})"


# --------------------------------------------------------------------------------------------
# Number formats and helpers
# --------------------------------------------------------------------------------------------

def check_e4m3_all_codes(lib):
    """Every one of the 256 e4m3fn codes decodes like torch's float8_e4m3fn cast."""
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    got = np.array([lib.oracle_e4m3_to_double(c) for c in range(256)])
    r = ref.numpy()
    assert (np.isnan(got) == np.isnan(r)).all()
    m = ~np.isnan(r)
    assert (got[m] == r[m]).all(), np.argwhere(got[m] != r[m])[:4]
    assert np.signbit(got[m]).tolist() == np.signbit(r[m]).tolist()  # -0 decodes to -0


def check_f32_le(lib):
    """The 4-byte scale decodes as little-endian binary32 (struct's '<f')."""
    for v in (1.0, -2.5, 0.3, 3.0e38, 1e-42, float("inf")):
        raw = struct.pack("<f", v)
        got = oracle.f32_le(raw, lib=lib)
        assert got == struct.unpack("<f", raw)[0], (v, got)


def check_helpers_worked_examples(lib):
    for ex in GOLDEN["min_block_table_width"]:
        assert oracle.min_block_table_width(ex["seq_len"], ex["block_size"], lib=lib) == ex["value"]
    # The pages state the helper as ceil(seq_len / block_size); the Example's other request
    # length 3000 at 32-token blocks needs ceil(93.75) = 94 entries.
    assert oracle.min_block_table_width(3000, 32, lib=lib) == 94
    assert oracle.min_block_table_width(1, 64, lib=lib) == 1
    assert oracle.min_block_table_width(0, 64, lib=lib) == 0
    for ex in GOLDEN["padded_seq_len"]:
        assert oracle.padded_seq_len(ex["max_seq_len"], lib=lib) == ex["value"]
    ex = GOLDEN["extents"]
    got = [oracle.row_end(ex["seq_len"], ex["next_n"], t, lib=lib) for t in range(ex["next_n"])]
    assert got == ex["row_ends"], got
    # A sequence shorter than the draft depth leaves its early slots empty.
    assert oracle.row_end(1, 3, 0, lib=lib) == 0 and oracle.row_end(1, 3, 2, lib=lib) == 1


# --------------------------------------------------------------------------------------------
# Logits
# --------------------------------------------------------------------------------------------

def check_layout_worked_block(lib):
    """A block laid out byte by byte at the offsets the pages print (bs=32, hd=128: values of
    token i at i*128, its scale at 4096 + 4*i, 4224 bytes a block).  With q = one-hot on dim d0
    in head 0 and weight 1 on head 0 only, logit[p] = scale[p] * max(k_p[d0], 0) exactly."""
    g = GOLDEN["kv_fused_block"]
    bs, D = g["block_size"], g["head_dim"]
    stride, s0, nbytes = g["token_value_stride"], g["scales_start"], g["block_bytes"]
    rng = np.random.default_rng(5)
    num_blocks, L = 3, 80
    vals = rng.standard_normal((num_blocks, bs, D)).astype(np.float32)
    codes = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    scales = rng.uniform(0.5, 2.0, (num_blocks, bs)).astype(np.float32)
    kv = np.zeros((num_blocks, nbytes), dtype=np.uint8)
    for blk in range(num_blocks):
        for i in range(bs):
            kv[blk, g["values_start"] + i * stride: g["values_start"] + i * stride + D] = codes[blk, i]
            kv[blk, s0 + 4 * i: s0 + 4 * i + 4] = np.frombuffer(struct.pack("<f", scales[blk, i]),
                                                                dtype=np.uint8)
    # The pages' torch.cat recipe gives the same bytes.
    cat = torch.cat([torch.from_numpy(codes).flatten(1),
                     torch.from_numpy(scales).view(torch.uint8).flatten(1)], dim=1).numpy()
    assert (cat == kv).all()
    H, d0 = 4, 17
    q = np.zeros((1, 1, H, D), dtype=np.uint8)
    q[0, 0, 0, d0] = 0x38                                   # e4m3 1.0
    weights = np.zeros((1, H), dtype=np.float32)
    weights[0, 0] = 1.0
    weights[0, 1:] = -0.75                                  # heads whose q is zero add nothing
    bt = np.array([[2, 0, 1]], dtype=np.int32)
    out, _ = oracle.paged_logits(q, kv, weights, bt, np.array([L], np.int32), 96, block_size=bs,
                                 lib=lib)
    kdec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for p in range(L):
        blk, i = bt[0, p // bs], p % bs
        want = float(scales[blk, i]) * max(kdec[blk, i, d0], 0.0)
        assert out[0, p] == want, (p, out[0, p], want)
    assert np.isnan(out[0, L:]).all()


def check_dense_matmul(lib):
    """Brute force: torch float64 matmul on de-paged K, several shapes, next_n 1..4, a zero-length
    request and one shorter than next_n."""
    cases = [
        _small(),
        _small(seed=12, batch=4, next_n=1, lens=(64, 0, 1, 200), max_seq_len=256, block_size=64,
               heads=16, head_dim=128),
        _small(seed=13, batch=2, next_n=4, lens=(3, 130), max_seq_len=192, block_size=64,
               heads=64, head_dim=128),
        _small(seed=14, batch=2, next_n=2, lens=(127, 128), max_seq_len=128, block_size=128,
               heads=4, head_dim=64, scale_range=(0.25, 4.0), outlier_frac=0.05),
    ]
    for w in cases:
        got, tol = _logits(lib, w)
        ref = dense_reference(w)
        _same(got, ref, rtol=1e-12, scale=np.where(np.isnan(tol), 0, tol))


def check_relu_per_head(lib):
    """ReLU before the weighted sum: negating q swaps relu(s) for relu(-s), and
    relu(x) - relu(-x) = x, so logits(q) - logits(-q) = scale[p] * sum_h w_h (q_h . k_p), which
    is linear and computed here with a float64 matmul.  Also: with U[-1,1] weights some logits
    are negative, and with |w| none is."""
    w = _small(seed=21, batch=2, next_n=2, lens=(90, 41), max_seq_len=96)
    a, tol = _logits(lib, w)
    qneg = w.q.clone()
    qneg ^= 0x80                                            # flip every e4m3 sign bit
    wn = synth.Workload(**{**w.__dict__, "q": qneg})
    b_, _ = _logits(lib, wn)
    diff = a - b_
    ref = np.full_like(a, np.nan)
    bs, D = w.block_size, w.head_dim
    vals = (w.kv_fused[:, :bs * D].contiguous().view(torch.float8_e4m3fn)
            .view(-1, bs, D).to(torch.float64))
    scl = w.kv_fused[:, bs * D:].contiguous().view(torch.float32).view(-1, bs).to(torch.float64)
    q = w.q.view(torch.float8_e4m3fn).to(torch.float64)
    for bi in range(w.batch):
        L = int(w.seq_lens[bi])
        pages = w.block_tables[bi, :math.ceil(L / bs)].long()
        K = vals[pages].reshape(-1, D)[:L]
        S = scl[pages].reshape(-1)[:L]
        for t in range(w.next_n):
            re = L - w.next_n + t + 1
            r = bi * w.next_n + t
            lin = (w.weights[r].double() @ q[bi, t]) @ K[:re].T
            ref[r, :re] = (S[:re] * lin).numpy()
    _same(diff, ref, rtol=1e-11, scale=np.where(np.isnan(tol), 0, 2 * tol + np.abs(ref)))
    assert np.nanmin(a) < 0.0
    wp = synth.Workload(**{**w.__dict__, "weights": w.weights.abs()})
    c, _ = _logits(lib, wp)
    assert np.nanmin(c) >= 0.0


def check_scale_linear(lib):
    """Doubling every per-token scale doubles every logit exactly; the tolerance magnitude is
    |scale| * sum_h |w_h relu(s_h)| and so doubles too."""
    w = _small(seed=31)
    a, ta = _logits(lib, w)
    bs, D = w.block_size, w.head_dim
    kv2 = w.kv_fused.clone()
    sc = kv2[:, bs * D:].contiguous().view(torch.float32) * 2.0
    kv2[:, bs * D:] = sc.view(torch.uint8)
    b_, tb = _logits(lib, synth.Workload(**{**w.__dict__, "kv_fused": kv2}))
    _same(b_, 2.0 * a, rtol=0.0)
    _same(tb, 2.0 * ta, rtol=0.0)


def check_paging_metamorphic(lib):
    """Moving pages to other physical blocks (and the table with them) changes nothing; the
    oracle never reads a table entry past a request's own page count (poison there is fine);
    an entry it needs that points outside the pool is an error."""
    w = _small(seed=41, batch=3, next_n=2, lens=(100, 33, 64), max_seq_len=128, pool_pages=12,
               unused_entries="poison")
    a, _ = _logits(lib, w)
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(3))
    kv2 = torch.empty_like(w.kv_fused)
    kv2[perm] = w.kv_fused                                   # block i moves to perm[i]
    bt2 = w.block_tables.clone()
    used = bt2 != 0x7FFFFFFF
    bt2[used] = perm[bt2[used].long()].to(torch.int32)
    b_, _ = _logits(lib, synth.Workload(**{**w.__dict__, "kv_fused": kv2, "block_tables": bt2}))
    _same(b_, a, rtol=0.0)
    bad = w.block_tables.clone()
    bad[1, 0] = w.num_blocks
    try:
        _logits(lib, synth.Workload(**{**w.__dict__, "block_tables": bad}))
    except oracle.OracleError as e:
        assert "-2" in str(e)
    else:
        raise AssertionError("an out-of-pool page was read without an error")


def check_extents(lib):
    """Exactly positions 0 .. seq_len - next_n + t are written in row b*next_n + t; rows of a
    zero-length request are not written at all."""
    w = _small(seed=51, batch=4, next_n=3, lens=(10, 0, 2, 64), max_seq_len=64)
    a, _ = _logits(lib, w, fill=np.nan)
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        for t in range(w.next_n):
            row = a[b * w.next_n + t]
            want = max(0, L - w.next_n + t + 1)
            written = ~np.isnan(row)
            assert written.sum() == want and written[:want].all(), (b, t, written.sum(), want)


# --------------------------------------------------------------------------------------------
# Top-k and the select contract
# --------------------------------------------------------------------------------------------

def check_total_order(lib):
    """IEEE totalOrder on a hand-ordered list (-NaN < -inf < -1 < -0 < +0 < tiny < 1 < inf <
    +NaN)."""
    neg_nan = struct.unpack("<f", struct.pack("<I", 0xFFC00000))[0]
    pos_nan = struct.unpack("<f", struct.pack("<I", 0x7FC00000))[0]
    seq = [neg_nan, -math.inf, -1.0, -0.0, 0.0, 1e-45, 1.0, math.inf, pos_nan]
    for i, a in enumerate(seq):
        for j, b in enumerate(seq):
            c = oracle.total_order_cmp(a, b, lib=lib)
            assert (c > 0) - (c < 0) == (i > j) - (i < j), (a, b, c)


def check_topk_distinct(lib):
    """Distinct values: torch.topk (sorted) gives the same indices in the same order."""
    g = torch.Generator().manual_seed(61)
    x = torch.randn(6, 300, generator=g)
    row_ends = torch.tensor([300, 7, 0, 64, 299, 150], dtype=torch.int32)
    idx, cnt = oracle.topk(x, row_ends, 64, lib=lib)
    for r in range(6):
        n = int(row_ends[r])
        k = min(n, 64)
        assert cnt[r] == k
        if k:
            ref = torch.topk(x[r, :n], k, sorted=True).indices.numpy()
            assert (idx[r, :k] == ref).all(), r


def check_topk_ties(lib):
    """Many equal values: numpy.lexsort by (-value, index) gives the same selection."""
    g = torch.Generator().manual_seed(62)
    x = torch.randint(0, 5, (4, 200), generator=g).to(torch.float32)
    row_ends = torch.tensor([200, 199, 3, 100], dtype=torch.int32)
    idx, cnt = oracle.topk(x, row_ends, 37, lib=lib)
    for r in range(4):
        n = int(row_ends[r])
        v = x[r, :n].numpy()
        order = np.lexsort((np.arange(n), -v))[:min(n, 37)]
        assert (idx[r, :cnt[r]] == order).all(), r


def check_slots_worked(lib):
    s = GOLDEN["slots"]
    cs = [oracle.slot_of(True, n, s["top_k"], s["capacity"], lib=lib)
          for n in range(len(s["candidate_slots"]))]
    ts = [oracle.slot_of(False, n, s["top_k"], s["capacity"], lib=lib)
          for n in range(len(s["tie_slots"]))]
    assert cs == s["candidate_slots"] and ts == s["tie_slots"], (cs, ts)


def _stored_topk(x_row, n, thr, top_k, capacity, k, arrival):
    """The top-k taken from what a row's slots would hold: keys arrive in the order ``arrival``
    (a permutation, standing in for the GPU's unspecified order); the first ``capacity``
    candidates and the first ``top_k`` ties get slots.  Ordered by value desc then index asc."""
    v = x_row[:n]
    order_in = arrival[arrival < n]
    cand = [i for i in order_in if v[i] > thr][:capacity]
    tie = [i for i in order_in if not (v[i] > thr) and not (v[i] < thr)][:top_k]
    items = np.array(cand + tie, dtype=np.int64)
    order = np.lexsort((items, -v[items]))
    return items[order][:k]


def check_classify_closed_forms(lib):
    """thr=+inf: no candidates; thr=-inf: every finite key is a candidate; thr=NaN: every key
    is a tie; thr = the K'-th largest of distinct values: K'-1 candidates and 1 tie, which fits
    (the select's description: a threshold at its top_k-th largest score makes a row fit)."""
    g = torch.Generator().manual_seed(71)
    x = torch.randn(3, 500, generator=g)
    x[1, 10] = math.inf
    x[2, 20] = math.nan
    re = torch.tensor([500, 500, 400], dtype=torch.int32)
    top_k, cap = 64, 63
    inf = torch.full((3,), math.inf)
    nc, nt, fits = oracle.select_classify(x, re, inf, top_k, cap, lib=lib)
    assert nc.tolist() == [0, 0, 0] and nt.tolist() == [0, 1, 1], (nc, nt)
    assert not fits.any()
    nc, nt, fits = oracle.select_classify(x, re, -inf, top_k, cap, lib=lib)
    assert nc.tolist() == [500, 500, 399] and nt.tolist() == [0, 0, 1]
    nc, nt, fits = oracle.select_classify(x, re, torch.full((3,), math.nan), top_k, cap, lib=lib)
    assert nc.tolist() == [0, 0, 0] and nt.tolist() == [500, 500, 400]
    kth = torch.stack([torch.sort(x[0, :500], descending=True).values[top_k - 1],
                       torch.sort(x[1, :500], descending=True).values[top_k - 1],
                       torch.sort(x[2, :400][~torch.isnan(x[2, :400])],
                                  descending=True).values[top_k - 1]])
    nc, nt, fits = oracle.select_classify(x, re, kth, top_k, cap, lib=lib)
    assert nc.tolist() == [top_k - 1, top_k - 1, top_k - 1], nc
    assert nt.tolist() == [1, 1, 2], nt                    # row 2's NaN is also a tie
    assert fits.all()


def check_fit_rule_gives_topk(lib):
    """Whenever the oracle says a row fits, its stored candidates and ties contain the row's
    exact top-K' (ties by lowest index), which torch.topk / numpy.lexsort confirm; with capacity
    >= top_k - 1 a threshold at or a little below the K'-th largest value always fits."""
    g = torch.Generator().manual_seed(81)
    rows, n, top_k, cap = 60, 400, 32, 40
    x = torch.randint(-20, 20, (rows, n), generator=g).to(torch.float32) / 4.0
    x[:10, :] = 1.5                                          # rows made of one repeated value
    x[10:20, ::2] = 0.25                                     # and rows full of one tie value
    re = torch.randint(0, n + 1, (rows,), generator=g).to(torch.int32)
    thr = torch.randint(-24, 24, (rows,), generator=g).to(torch.float32) / 4.0
    thr[:10] = 1.5
    thr[10:20] = 0.25
    nc, nt, fits = oracle.select_classify(x, re, thr, top_k, cap, lib=lib)
    assert fits.any() and not fits.all()
    for r in range(rows):
        k = min(int(re[r]), top_k)
        v = x[r].numpy()
        ref = np.lexsort((np.arange(int(re[r])), -v[:int(re[r])]))[:k]
        if fits[r]:
            arrival = np.random.default_rng(r).permutation(n)
            got = _stored_topk(v, int(re[r]), float(thr[r]), top_k, cap, k, arrival)
            assert (np.sort(got) == np.sort(ref)).all(), r
    kth = torch.tensor([float(x[r, :int(re[r])].sort(descending=True).values[min(int(re[r]), top_k) - 1])
                        if int(re[r]) else 0.0 for r in range(rows)])
    _, nt2, fits2 = oracle.select_classify(x, re, kth, top_k, top_k - 1, lib=lib)
    # At its K'-th largest value a row fits whenever every tie it needs has a slot.
    assert fits2[nt2 <= top_k].all() and (nt2 <= top_k).sum() >= rows // 2


# --------------------------------------------------------------------------------------------
# Schedule
# --------------------------------------------------------------------------------------------

def check_schedule_invariants(lib):
    """Expanding every CTA's [start, next start) range visits each (request, tile) unit exactly
    once, in order, and the ranges' sizes differ by at most one."""
    g = torch.Generator().manual_seed(91)
    for trial in range(6):
        B = int(torch.randint(1, 40, (1,), generator=g))
        lens = torch.randint(0, 3000, (B,), generator=g).to(torch.int32)
        lens[torch.rand(B, generator=g) < 0.2] = 0
        ctas = int(torch.randint(1, 200, (1,), generator=g))
        tile = 128
        sched = oracle.schedule(lens, tile, ctas, lib=lib)
        units = [(b, j) for b in range(B) for j in range(-(-int(lens[b]) // tile))]
        pos = {u: i for i, u in enumerate(units)}
        pos[(B, 0)] = len(units)
        starts = [pos[(int(s[0]), int(s[1]))] for s in sched]
        assert starts[0] == 0 and starts[-1] == len(units), (starts[0], starts[-1])
        sizes = np.diff(starts)
        assert (sizes >= 0).all() and sizes.max() - sizes.min() <= 1, sizes


# --------------------------------------------------------------------------------------------
# MXFP4 ("flashinfer.attn_scores", fp4_paged_mqa_logits)
# --------------------------------------------------------------------------------------------

# The FP4 E2M1 element values by code (OCP Microscaling Formats specification v1.0, the E2M1
# table): codes 0-7 are +0, 0.5, 1, 1.5, 2, 3, 4, 6; codes 8-15 the same with the sign set.
OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def check_e2m1_codes(lib):
    got = [lib.oracle_e2m1_to_double(c) for c in range(16)]
    assert got[:8] == OCP_E2M1, got[:8]
    assert got[8:] == [-v for v in OCP_E2M1], got[8:]
    assert math.copysign(1.0, got[8]) < 0  # code 8 is -0


def check_ue8m0_vs_torch(lib):
    """All 256 scale bytes against torch's float8_e8m0fnu decode (2^(e - 127), 0xFF NaN)."""
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu)
    ref = ref.to(torch.float64).tolist()
    for e in range(256):
        got = lib.oracle_ue8m0_to_double(e)
        assert (math.isnan(got) and math.isnan(ref[e])) or got == ref[e], (e, got, ref[e])


def _mx_single(lib, q_vals, q_sf, block, block_size, head_dim, seq_len, weights):
    """One request, one head, one page: the oracle's MXFP4 logits row."""
    q = np.asarray(q_vals, dtype=np.uint8).reshape(1, 1, 1, head_dim // 2)
    qsf = np.asarray(q_sf, dtype=np.uint8).reshape(1, 1, 1, head_dim // 32)
    kv = np.asarray(block, dtype=np.uint8).reshape(1, -1)
    bt = np.zeros((1, 1), dtype=np.int32)
    sl = np.array([seq_len], dtype=np.int32)
    w = np.asarray(weights, dtype=np.float32).reshape(1, 1)
    out, _ = oracle.paged_logits_mxfp4(q, qsf, kv, w, bt, sl, seq_len, block_size=block_size,
                                       lib=lib)
    return out[0]


def check_mxfp4_layout_worked_block(lib):
    """The pages' drawing for block_size 32, head_dim 128: token i's 64 packed bytes at i*64,
    its 4 scale bytes at 2048 + 4*i (byte k for elements [32k, 32k+32)); byte j holds element 2j
    in the low nibble and 2j+1 in the high nibble.  A block written byte by byte at those offsets
    with one nonzero element per token must give w * q_d * k_d * 2^(e - 127) at each token."""
    ex = GOLDEN["mxfp4_block"]
    BS, D = ex["block_size"], ex["head_dim"]
    assert ex["values_bytes"] == BS * D // 2 and ex["scale_offset_token_1"] == BS * D // 2 + 4
    for d0 in (0, 1, 37, 127):
        q = np.zeros(D // 2, dtype=np.uint8)
        q[d0 // 2] = 2 << (4 * (d0 % 2))          # q element d0 = code 2 = 1.0
        q_sf = [127] * (D // 32)                   # 2^0
        block = np.zeros(BS * (D // 2 + D // 32), dtype=np.uint8)
        expect = []
        for i in range(BS):
            code = 1 + i % 7                       # 0.5 .. 6
            e = 120 + i % 9                        # 2^-7 .. 2^1
            block[i * 64 + d0 // 2] = code << (4 * (d0 % 2))
            block[2048 + 4 * i + d0 // 32] = e
            expect.append(OCP_E2M1[code] * 2.0 ** (e - 127) * 0.75)
        got = _mx_single(lib, q, q_sf, block, BS, D, BS, [0.75])
        assert np.array_equal(got[:BS], np.array(expect)), (d0, got[:4], expect[:4])


def check_mxfp4_matches_fp8(lib):
    """With every scale byte 127 (2^0) the MXFP4 logits equal the FP8 oracle's (per-token scale
    1.0) on the same element values, which e4m3 represents exactly; scaling all of a K token's
    scale bytes by 2^e equals a per-token scale of 2^e there, and all of a q head's by 2^a a
    weight scaled by 2^a (a positive power of two commutes with the ReLU).  Both sums are
    exact, so the results agree bit for bit."""
    g = torch.Generator().manual_seed(404)
    B, n, H, D, BS = 2, 2, 4, 64, 32
    lens = [70, 33]
    w = synth.make_workload("mx", 21, B, n, 96, "fixed", values=lens, num_heads=H, head_dim=D,
                            block_size=BS)
    pool = w.num_blocks
    qc = torch.randint(0, 16, (B, n, H, D), generator=g)
    kc = torch.randint(0, 16, (pool, BS, D), generator=g)
    table = torch.tensor(OCP_E2M1 + [-v for v in OCP_E2M1], dtype=torch.float32)
    pack = lambda c: (c[..., 0::2] | (c[..., 1::2] << 4)).to(torch.uint8)
    kexp = torch.randint(-3, 4, (pool, BS), generator=g)
    qexp = torch.randint(-2, 3, (B, n, H), generator=g)
    qm = pack(qc)
    qsf = (127 + qexp)[..., None].expand(B, n, H, D // 32).to(torch.uint8).contiguous()
    ksf = (127 + kexp)[..., None].expand(pool, BS, D // 32).to(torch.uint8)
    kv4 = torch.cat([pack(kc).flatten(1), ksf.flatten(1)], dim=1).contiguous()
    out4, _ = oracle.paged_logits_mxfp4(qm, qsf, kv4, w.weights, w.block_tables, w.seq_lens,
                                        w.max_seq_len, block_size=BS, lib=lib)
    q8 = table[qc].to(torch.float8_e4m3fn).view(torch.uint8)
    k8 = table[kc].to(torch.float8_e4m3fn).view(torch.uint8)
    scale = torch.exp2(kexp.to(torch.float32))
    kv8 = torch.cat([k8.flatten(1), scale.view(torch.uint8).flatten(1)], dim=1).contiguous()
    w8 = (w.weights * torch.exp2(qexp.to(torch.float32)).reshape(B * n, H)).contiguous()
    out8, _ = oracle.paged_logits(q8.contiguous(), kv8, w8, w.block_tables, w.seq_lens,
                                  w.max_seq_len, block_size=BS, lib=lib)
    assert np.array_equal(np.nan_to_num(out4, nan=-7.0), np.nan_to_num(out8, nan=-7.0))


ALL_CHECKS = [
    check_e4m3_all_codes, check_f32_le, check_helpers_worked_examples, check_layout_worked_block,
    check_dense_matmul, check_relu_per_head, check_scale_linear, check_paging_metamorphic,
    check_extents, check_total_order, check_topk_distinct, check_topk_ties, check_slots_worked,
    check_classify_closed_forms, check_fit_rule_gives_topk, check_schedule_invariants,
    check_e2m1_codes, check_ue8m0_vs_torch, check_mxfp4_layout_worked_block,
    check_mxfp4_matches_fp8,
]
