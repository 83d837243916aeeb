"""MXFP4 paged logits: the CUDA path (staging + FP8 logits kernel) against the float64 MXFP4
oracle, element by element, with the logits tolerance of the FP8 path."""
import numpy as np
import pytest
import torch

import oracle
import paged_fp8_mqa_gb300 as idx
from paged_fp8_mqa_gb300 import synth
from gpu_cases import check_logits, expected_row_ends, expected_scores

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    idx.device_status(clear=True)
    yield
    assert idx.device_status(clear=True) == 0, "a kernel raised a device status bit"


def _case(seed, next_n, lens, heads=64, head_dim=128, block_size=64, spread=0):
    w = synth.make_workload("mxfp4", seed, len(lens), next_n, max(max(lens), 1), "fixed",
                            values=list(lens), num_heads=heads, head_dim=head_dim,
                            block_size=block_size)
    return w, synth.make_mxfp4(w, spread_tokens=spread)


def _oracle(w, m):
    return oracle.paged_logits_mxfp4(m.q, m.q_sf, m.kv_fused, w.weights, w.block_tables,
                                     w.seq_lens, w.max_seq_len, block_size=w.block_size)


def _gpu(w, m, dtype=torch.float32, num_sms=0):
    d = torch.device("cuda:0")
    out = torch.full((w.rows, idx.idx_padded_seq_len(w.max_seq_len)), float("nan"), dtype=dtype,
                     device=d)
    row_ends = torch.full((w.rows,), -7, dtype=torch.int32, device=d)
    idx.logits_mxfp4(m.q.to(d), m.q_sf.to(d), m.kv_fused.to(d), w.weights.to(d),
                     w.block_tables.to(d), w.seq_lens.to(d), w.max_seq_len, out=out,
                     row_ends_out=row_ends, num_sms=num_sms)
    torch.cuda.synchronize()
    return out, row_ends


CASES = [
    (1, 64, 128, 64, [5000, 1, 0, 777, 129]),
    (2, 64, 128, 32, [3000, 0, 2, 64, 65, 4097]),
    (3, 32, 128, 128, [2500, 3, 2, 0, 127, 129]),
    (4, 64, 64, 64, [4000, 4, 3, 100, 0, 8193]),
    (2, 32, 64, 32, [3000, 1, 0, 200, 7000]),
    (3, 64, 128, 64, [2900, 2, 0, 131, 6001]),
]


@pytest.mark.parametrize("next_n,heads,head_dim,block_size,lens", CASES,
                         ids=[f"n{n}-h{h}-d{d}-bs{b}" for n, h, d, b, _ in CASES])
def test_mxfp4_parity(next_n, heads, head_dim, block_size, lens):
    w, m = _case(600 + next_n + heads + head_dim, next_n, lens, heads, head_dim, block_size)
    ref, tol = _oracle(w, m)
    got, row_ends = _gpu(w, m)
    stats = check_logits(w, got, ref, tol)
    assert stats["checked"] == expected_scores(w)
    assert (row_ends.cpu().numpy() == expected_row_ends(w)).all()


@pytest.mark.parametrize("next_n", [1, 3, 4])
def test_mxfp4_one_cta_many_lists(next_n):
    """One CTA walks several tile lists of many short requests: the converter groups take the
    run's tiles in turn across list boundaries."""
    g = torch.Generator().manual_seed(45 + next_n)
    lens = torch.randint(1, 700, (120,), generator=g).tolist()
    w, m = _case(650 + next_n, next_n, lens)
    ref, tol = _oracle(w, m)
    got, row_ends = _gpu(w, m, num_sms=1)
    stats = check_logits(w, got, ref, tol)
    assert stats["checked"] == expected_scores(w)
    assert (row_ends.cpu().numpy() == expected_row_ends(w)).all()


def test_mxfp4_long_runs_and_float16():
    """One CTA over several tile lists; float16 output equals the float32 result rounded."""
    g = torch.Generator().manual_seed(44)
    lens = torch.randint(1, 900, (100,), generator=g).tolist()
    w, m = _case(640, 2, lens)
    ref, tol = _oracle(w, m)
    got, _ = _gpu(w, m, num_sms=1)
    check_logits(w, got, ref, tol)
    got16, _ = _gpu(w, m, dtype=torch.float16)
    re = expected_row_ends(w)
    a, b = got.cpu(), got16.cpu()
    for r in range(w.rows):
        e = int(re[r])
        assert torch.equal(a[r, :e].to(torch.float16), b[r, :e]), f"row {r}"


def test_mxfp4_wide_scale_spread_is_flagged():
    """KV tokens whose block scales span more than 8 binades are staged with rounding and
    raise IDX_DEV_INEXACT_SCALE; the other positions stay exact."""
    w, m = _case(650, 1, [3000, 2000], spread=40)
    ref, tol = _oracle(w, m)
    got, _ = _gpu(w, m)
    status = idx.device_status(clear=True)
    assert status & idx.IDX_DEV_INEXACT_SCALE
    g = got.cpu().double().numpy()
    re = expected_row_ends(w)
    close = 0
    for r in range(w.rows):
        e = int(re[r])
        err = np.abs(g[r, :e] - ref[r, :e])
        close += int((err <= 2e-6 * tol[r, :e] + 1e-7).sum())
    assert close >= expected_scores(w) - 40  # only the spread tokens may differ


def test_mxfp4_bfloat16_output():
    """bfloat16 output (the pages' default for this variant; head_dim 128) equals the float32
    result rounded to nearest even."""
    w, m = _case(660, 2, [3000, 0, 700, 129], block_size=32)
    got, _ = _gpu(w, m)
    got_bf, _ = _gpu(w, m, dtype=torch.bfloat16)
    re = expected_row_ends(w)
    a, b = got.cpu(), got_bf.cpu()
    for r in range(w.rows):
        e = int(re[r])
        assert torch.equal(a[r, :e].to(torch.bfloat16), b[r, :e]), f"row {r}"


def test_mxfp4_bfloat16_refused_for_head_dim_64():
    w, m = _case(661, 1, [300], head_dim=64)
    with pytest.raises(idx.IdxError) as e:
        _gpu(w, m, dtype=torch.bfloat16)
    assert e.value.status == idx.IDX_UNSUPPORTED


@pytest.mark.parametrize("byte", [254, 250, 1, 0])
def test_mxfp4_extreme_q_scale_is_flagged(byte):
    """A q row whose largest scale byte moves its weight out of float32's normal range (the
    weight times 2^(E - 127) overflows or turns subnormal) raises IDX_DEV_INEXACT_SCALE; rows of
    ordinary scales are unaffected."""
    w, m = _case(670 + byte, 1, [600, 900])
    q_sf = m.q_sf.clone()
    q_sf[1, 0, 5, :] = byte  # request 1, head 5: every group at the extreme byte
    weights = w.weights.clone()
    weights[1, 5] = 3.0e38 if byte >= 250 else 1.0e-30
    w2 = synth.Workload(**{**w.__dict__, "weights": weights})
    m2 = synth.Mxfp4Inputs(q=m.q, q_sf=q_sf, kv_fused=m.kv_fused)
    ref, tol = _oracle(w2, m2)
    got, _ = _gpu(w2, m2)
    assert idx.device_status(clear=True) & idx.IDX_DEV_INEXACT_SCALE
    g = got.cpu().double().numpy()
    e = int(expected_row_ends(w2)[0])  # request 0 is untouched by the extreme head
    assert (np.abs(g[0, :e] - ref[0, :e]) <= 2e-6 * tol[0, :e] + 1e-7).all()
