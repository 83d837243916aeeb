"""Paged FP8 MQA logits: the CUDA path against the float64 oracle, element by element."""
import numpy as np
import pytest
import torch

import oracle
import paged_fp8_mqa_gb300 as idx
from paged_fp8_mqa_gb300 import synth
from gpu_cases import (check_logits, gpu_logits, oracle_logits_cached, to_device, expected_row_ends, expected_scores)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    idx.device_status(clear=True)
    yield
    assert idx.device_status(clear=True) == 0, "a kernel raised a device status bit"


def _small(seed, next_n, lens, max_seq_len=None, **kw):
    m = max_seq_len or max(max(lens), 1)
    return synth.make_workload("edge", seed, len(lens), next_n, m, "fixed", values=list(lens),
                               **kw)


def _oracle(w):
    return oracle.paged_logits(w.q, w.kv_fused, w.weights, w.block_tables, w.seq_lens,
                               w.max_seq_len, block_size=w.block_size)


def test_tiny_workload():
    w, ref, tol = oracle_logits_cached("tiny")
    got, row_ends = gpu_logits(w)
    check_logits(w, got, ref, tol)
    assert (row_ends.cpu().numpy() == expected_row_ends(w)).all()


EDGE = [
    (1, [1]), (1, [63]), (1, [64]), (1, [65]), (1, [127, 128, 129]), (1, [255, 256, 257]),
    (2, [1, 2, 3]), (2, [0, 64, 0, 130]), (3, [2, 3, 4, 200]), (4, [3, 4, 5, 1000]),
    (4, [0, 0, 0]), (1, [5000, 1, 0, 77]), (3, [129, 64, 63, 1]), (2, [4096, 4095]),
]


@pytest.mark.parametrize("next_n,lens", EDGE, ids=[f"n{n}-{'_'.join(map(str, l))}" for n, l in EDGE])
def test_edge_lengths(next_n, lens):
    w = _small(100 + len(lens) + next_n, next_n, lens)
    ref, tol = _oracle(w)
    got, row_ends = gpu_logits(w)
    check_logits(w, got, ref, tol)
    assert (row_ends.cpu().numpy() == expected_row_ends(w)).all()


@pytest.mark.parametrize("next_n", [1, 2, 3, 4])
def test_many_requests_ragged(next_n):
    g = torch.Generator().manual_seed(next_n)
    lens = torch.randint(0, 3000, (37,), generator=g).tolist()
    w = _small(200 + next_n, next_n, lens, max_seq_len=3000, scale_range=(0.25, 4.0),
               outlier_frac=0.01)
    ref, tol = _oracle(w)
    got, _ = gpu_logits(w)
    check_logits(w, got, ref, tol)


@pytest.mark.parametrize("num_sms", [1, 3, 37, 500])
def test_grid_size_does_not_change_results(num_sms):
    w = _small(301, 2, [700, 0, 1300, 64, 65, 2000])
    base, _ = gpu_logits(w)
    got, _ = gpu_logits(w, num_sms=num_sms)
    assert torch.equal(got.nan_to_num(-1e30), base.nan_to_num(-1e30))


def test_precomputed_schedule_matches_in_kernel_split():
    w = _small(302, 3, [900, 5, 0, 4000, 128])
    base, _ = gpu_logits(w)
    got, _ = gpu_logits(w, schedule=True)
    assert torch.equal(got.nan_to_num(-1e30), base.nan_to_num(-1e30))
    for n_sms in (1, 10, 152):
        got2, _ = gpu_logits(w, schedule=True, num_sms=n_sms)
        assert torch.equal(got2.nan_to_num(-1e30), base.nan_to_num(-1e30))


def test_strided_table_and_lengths():
    """block_tables[::2] and seq_lens[::2] views are read without a copy."""
    w = _small(303, 2, [300, 1000, 17])
    t = to_device(w)
    B, W = w.block_tables.shape
    bt2 = torch.full((2 * B, W), 0x7FFFFFFF, dtype=torch.int32, device=t["bt"].device)
    bt2[::2] = t["bt"]
    sl2 = torch.full((2 * B,), 999999, dtype=torch.int32, device=t["bt"].device)
    sl2[::2] = t["seq_lens"]
    ref, tol = _oracle(w)
    got, _ = gpu_logits(w, tensors=t, bt=bt2[::2], seq_lens=sl2[::2])
    check_logits(w, got, ref, tol)


def test_unused_table_entries_never_read():
    w = _small(304, 1, [70, 300, 1], max_seq_len=1024, unused_entries="poison")
    ref, tol = _oracle(w)
    got, _ = gpu_logits(w)
    check_logits(w, got, ref, tol)


@pytest.mark.parametrize("name", ["decode", "mtp", "long_select", "serving"])
def test_full_workload(name):
    w, ref, tol = oracle_logits_cached(name)
    got, row_ends = gpu_logits(w)
    stats = check_logits(w, got, ref, tol)
    assert stats["checked"] == expected_scores(w)
    assert (row_ends.cpu().numpy() == expected_row_ends(w)).all()


@pytest.mark.parametrize("num_sms", [1, 2])
def test_runs_longer_than_one_tile_list(num_sms):
    """With one or two CTAs each CTA's run spans several tile lists (of at most 256 tiles)."""
    w = _small(305, 2, [40000, 30000, 5, 0, 7000], max_seq_len=40000)
    ref, tol = _oracle(w)
    got, _ = gpu_logits(w, num_sms=num_sms)
    check_logits(w, got, ref, tol)


@pytest.mark.parametrize("next_n", [1, 3])
def test_many_short_requests_over_several_tile_lists(next_n):
    """One CTA's run of ~300 requests of one to three tiles spans three tile lists: the q/w
    buffers, reused every second request, are released exactly once per request across the
    lists' boundaries (each list's first tile is a continued or a new request)."""
    g = torch.Generator().manual_seed(40 + next_n)
    lens = torch.randint(1, 330, (300,), generator=g).tolist()
    lens[100:110] = [0] * 10
    w = _small(307 + next_n, next_n, lens)
    ref, tol = _oracle(w)
    for num_sms in (1, 2):
        got, _ = gpu_logits(w, num_sms=num_sms)
        check_logits(w, got, ref, tol)


HEADS32 = [
    (1, 64, [5000, 1, 0, 777, 129, 64, 65]),
    (2, 32, [3000, 0, 2, 31, 33, 9000]),
    (3, 128, [2500, 3, 2, 0, 127, 129, 6000]),
    (4, 64, [4000, 4, 3, 100, 0, 8191, 8193]),
]


@pytest.mark.parametrize("next_n,block_size,lens", HEADS32,
                         ids=[f"n{n}-bs{b}" for n, b, _ in HEADS32])
def test_32_heads(next_n, block_size, lens):
    """num_heads = 32: MMA N = 32 * next_n, a thread holds 8 of the heads per slot."""
    w = _small(320 + next_n, next_n, lens, num_heads=32, block_size=block_size)
    ref, tol = _oracle(w)
    got, row_ends = gpu_logits(w)
    check_logits(w, got, ref, tol)
    assert (row_ends.cpu().numpy() == expected_row_ends(w)).all()


def test_32_heads_long_runs_and_float16():
    """num_heads = 32 over runs of several tile lists (one CTA), and with float16 output."""
    g = torch.Generator().manual_seed(32)
    lens = torch.randint(1, 900, (120,), generator=g).tolist()
    w = _small(330, 2, lens, num_heads=32)
    ref, tol = _oracle(w)
    got, _ = gpu_logits(w, num_sms=1)
    check_logits(w, got, ref, tol)
    t = to_device(w)
    out = torch.full((w.rows, idx.idx_padded_seq_len(w.max_seq_len)), float("nan"),
                     dtype=torch.float16, device="cuda")
    idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len, out=out)
    torch.cuda.synchronize()
    _check_float16(w, out, ref, tol)


DIM64 = [
    (1, 64, 64, [5000, 1, 0, 777, 129, 64, 65]),
    (2, 64, 32, [3000, 0, 2, 31, 33, 9000]),
    (3, 64, 128, [2500, 3, 2, 0, 127, 129, 6000]),
    (4, 64, 64, [4000, 4, 3, 100, 0, 8191, 8193]),
    (2, 32, 64, [3000, 1, 0, 200, 7000]),
    (4, 32, 128, [2000, 4, 0, 129, 5000]),
]


@pytest.mark.parametrize("next_n,heads,block_size,lens", DIM64,
                         ids=[f"n{n}-h{h}-bs{b}" for n, h, b, _ in DIM64])
def test_head_dim_64(next_n, heads, block_size, lens):
    """head_dim = 64: rows of 64 bytes, 64-byte swizzle, two K = 32 MMAs per tile."""
    w = _small(340 + next_n + heads, next_n, lens, num_heads=heads, head_dim=64,
               block_size=block_size)
    ref, tol = _oracle(w)
    got, row_ends = gpu_logits(w)
    check_logits(w, got, ref, tol)
    assert (row_ends.cpu().numpy() == expected_row_ends(w)).all()


def test_head_dim_64_long_runs_and_float16():
    g = torch.Generator().manual_seed(64)
    lens = torch.randint(1, 900, (120,), generator=g).tolist()
    w = _small(350, 3, lens, head_dim=64)
    ref, tol = _oracle(w)
    got, _ = gpu_logits(w, num_sms=1)
    check_logits(w, got, ref, tol)
    t = to_device(w)
    out = torch.full((w.rows, idx.idx_padded_seq_len(w.max_seq_len)), float("nan"),
                     dtype=torch.float16, device="cuda")
    idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len, out=out)
    torch.cuda.synchronize()
    _check_float16(w, out, ref, tol)


def test_stale_schedule_terminates():
    """A schedule computed for other lengths gives wrong coverage but no hang, no fault and no
    read past any request's pages."""
    w = _small(306, 1, [3000, 100, 9000, 64])
    t = to_device(w)
    other = torch.tensor([9000, 9000, 9000, 9000], dtype=torch.int32).cuda()
    stale = idx.schedule(other, 1, 8)
    pad = idx.idx_padded_seq_len(w.max_seq_len)
    out = torch.full((w.rows, pad), float("nan"), device="cuda")
    idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len, out=out,
                   schedule_meta=stale, num_sms=8)
    torch.cuda.synchronize()
    # Whatever was written is a correct logit: compare where the stale split reached.
    ref, tol = _oracle(w)
    got = out.cpu().double().numpy()
    m = ~np.isnan(got) & ~np.isnan(ref)
    assert (np.abs(got[m] - ref[m]) <= 2e-6 * tol[m] + 1e-7).all()


def _check_float16(w, out, ref, tol):
    """float16 output ("flashinfer.attn_scores", Parameters: output_dtype): the float32 result
    (within the float32 tolerance of the oracle) rounded to nearest even, so within that
    tolerance plus half a binary16 ulp of the value; values past the half range are +-inf (where
    the oracle's value is clear of the rounding boundary 65520 by more than the tolerance)."""
    got = out.cpu().double().numpy()
    re = expected_row_ends(w)
    lim32 = 2e-6 * tol + 1e-7
    for r in range(w.rows):
        L, e = int(w.seq_lens[r // w.next_n]), int(re[r])
        g, x, l32 = got[r, :e], ref[r, :e], lim32[r, :e]
        over = np.abs(x) - l32 >= 65520.0
        under = np.abs(x) + l32 < 65520.0
        assert (np.isinf(g[over]) & (np.sign(g[over]) == np.sign(x[over]))).all(), f"row {r}"
        a = np.abs(x[under]) + l32[under]
        half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -14))) - 11)
        err = np.abs(g[under] - x[under])
        assert (err <= l32[under] + half_ulp).all(), f"row {r}: max err {err.max()}"
        assert np.isnan(got[r, L:]).all(), f"row {r}: columns >= seq_len were written"


@pytest.mark.parametrize("next_n", [1, 2, 3, 4])
def test_float16_output(next_n):
    w = _small(310 + next_n, next_n, [1, 63, 64, 65, 300, 1000, 0, 4097], max_seq_len=4097)
    ref, tol = _oracle(w)
    t = to_device(w)
    pad = idx.idx_padded_seq_len(w.max_seq_len)
    out = torch.full((w.rows, pad), float("nan"), dtype=torch.float16, device="cuda")
    got = idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len,
                         out=out)
    torch.cuda.synchronize()
    assert got.dtype == torch.float16 and got.data_ptr() == out.data_ptr()
    _check_float16(w, out, ref, tol)


def test_float16_output_overflows_to_inf():
    """Weights scaled so that many logits leave the binary16 range."""
    w = _small(320, 2, [500, 130, 2000], max_seq_len=2000)
    w.weights.mul_(3000.0)
    ref, tol = _oracle(w)
    assert (np.abs(np.nan_to_num(ref)) > 70000).any()
    t = to_device(w)
    out = torch.full((w.rows, idx.idx_padded_seq_len(w.max_seq_len)), float("nan"),
                     dtype=torch.float16, device="cuda")
    idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len, out=out)
    torch.cuda.synchronize()
    _check_float16(w, out, ref, tol)


def test_output_dtype_keyword_allocates():
    w = _small(321, 1, [200, 5])
    t = to_device(w)
    got = idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len,
                         output_dtype=torch.float16)
    assert got.dtype == torch.float16 and got.shape == (w.rows, w.max_seq_len)
    with pytest.raises(ValueError):
        idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len,
                       out=torch.empty(w.rows, 256, device="cuda"), output_dtype=torch.float16)


BLOCK_LENS = [1, 31, 32, 33, 63, 64, 65, 127, 128, 129, 300, 0, 2049]


@pytest.mark.parametrize("block_size", [32, 128])
@pytest.mark.parametrize("next_n", [1, 2, 3, 4])
def test_block_sizes(block_size, next_n):
    """Pages of 32 or 128 tokens ("flashinfer.attn_scores", Parameters: kv_fused, block_size):
    a 128-position tile then spans four pages or one."""
    w = _small(330 + next_n + block_size, next_n, BLOCK_LENS, max_seq_len=2049,
               block_size=block_size)
    ref, tol = _oracle(w)
    got, row_ends = gpu_logits(w)
    check_logits(w, got, ref, tol)
    assert (row_ends.cpu().numpy() == expected_row_ends(w)).all()


@pytest.mark.parametrize("block_size", [32, 128])
def test_block_sizes_ragged_and_poisoned(block_size):
    """Many ragged requests with outlier keys; table entries past each request's pages hold an
    out-of-pool id that must never be read."""
    g = torch.Generator().manual_seed(block_size)
    lens = torch.randint(0, 5000, (41,), generator=g).tolist()
    w = _small(340 + block_size, 3, lens, max_seq_len=5000, block_size=block_size,
               scale_range=(0.25, 4.0), outlier_frac=0.01, unused_entries="poison")
    ref, tol = _oracle(w)
    got, _ = gpu_logits(w)
    check_logits(w, got, ref, tol)


def test_block_size_32_float16_output():
    w = _small(350, 4, [4000, 33, 1, 700], max_seq_len=4000, block_size=32)
    ref, tol = _oracle(w)
    t = to_device(w)
    out = torch.full((w.rows, idx.idx_padded_seq_len(w.max_seq_len)), float("nan"),
                     dtype=torch.float16, device="cuda")
    idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len, out=out)
    torch.cuda.synchronize()
    _check_float16(w, out, ref, tol)


@pytest.mark.parametrize("heads", [8, 16])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("next_n", [1, 2, 3, 4])
def test_few_heads(heads, head_dim, next_n):
    """8 and 16 heads ("flashinfer.attn_scores", fp8_paged_mqa_logits: num_heads % 4 == 0,
    next_n * num_heads in [8, 256]): the tensor core's N is next_n * heads rounded up to a
    multiple of 16 (8 heads at next_n 1 or 3 read extra q rows, or zeros past the end of q, into
    columns nobody reads).  Every page size, ragged lengths, the last request long."""
    for block_size in (32, 64, 128):
        w = _small(360 + heads + head_dim + next_n + block_size, next_n,
                   [0, 1, 129, 64, 300, 2049], max_seq_len=2049, num_heads=heads,
                   head_dim=head_dim, block_size=block_size)
        ref, tol = _oracle(w)
        got, row_ends = gpu_logits(w)
        check_logits(w, got, ref, tol)
        assert (row_ends.cpu().numpy() == expected_row_ends(w)).all()


@pytest.mark.parametrize("heads", [8, 16])
def test_few_heads_long_runs_and_float16(heads):
    """Many short requests over one to three CTAs (several tile lists each), and float16
    output equal to the float32 result rounded."""
    g = torch.Generator().manual_seed(heads)
    lens = torch.randint(0, 700, (160,), generator=g).tolist()
    w = _small(380 + heads, 3, lens, max_seq_len=700, num_heads=heads)
    ref, tol = _oracle(w)
    for num_sms in (1, 3):
        got, _ = gpu_logits(w, num_sms=num_sms)
        check_logits(w, got, ref, tol)
    t = to_device(w)
    out = torch.full((w.rows, idx.idx_padded_seq_len(w.max_seq_len)), float("nan"),
                     dtype=torch.float16, device="cuda")
    idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len, out=out)
    torch.cuda.synchronize()
    _check_float16(w, out, ref, tol)


@pytest.mark.parametrize("heads", [32, 64])
@pytest.mark.parametrize("next_n", [1, 2, 3, 4])
def test_head_dim_192(heads, next_n):
    """head_dim 192 ("flashinfer.attn_scores", fp8_paged_mqa_logits: head_dim % 32 == 0; the
    shared-memory note that 192 fits at 64 heads): each row three 64-byte K blocks, six MMAs per
    tile (scores may reach 192 * 448^2, above 2^25: the saturating ReLU rescale is 2^-26).  Every
    page size, ragged lengths, 2% of keys scaled x60 before the e4m3 cast."""
    for block_size in (32, 64, 128):
        w = _small(400 + heads + next_n + block_size, next_n, [0, 1, 129, 64, 300, 2049],
                   max_seq_len=2049, num_heads=heads, head_dim=192, block_size=block_size,
                   scale_range=(0.25, 4.0), outlier_frac=0.02, outlier_mult=60.0)
        ref, tol = _oracle(w)
        got, row_ends = gpu_logits(w)
        check_logits(w, got, ref, tol)
        assert (row_ends.cpu().numpy() == expected_row_ends(w)).all()


def test_head_dim_192_long_runs_and_float16():
    g = torch.Generator().manual_seed(192)
    lens = torch.randint(0, 900, (120,), generator=g).tolist()
    w = _small(420, 2, lens, max_seq_len=900, head_dim=192)
    ref, tol = _oracle(w)
    for num_sms in (1, 3, 0):
        got, _ = gpu_logits(w, num_sms=num_sms)
        check_logits(w, got, ref, tol)
    t = to_device(w)
    out = torch.full((w.rows, idx.idx_padded_seq_len(w.max_seq_len)), float("nan"),
                     dtype=torch.float16, device="cuda")
    idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len, out=out)
    torch.cuda.synchronize()
    _check_float16(w, out, ref, tol)
