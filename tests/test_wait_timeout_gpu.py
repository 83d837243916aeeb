"""The time-limited pipeline waits: a CTA made to withhold the copies of its first tile
(idx_debug_withhold_first_tile, test-only fault injection on the host's request) has every
wait on that tile run out after its one-second limit.  The launch must return, raise
IDX_DEV_WAIT_TIMEOUT, leave the context usable, and the other CTAs' scores must be right."""
import numpy as np
import pytest
import torch

import oracle
import paged_fp8_mqa_gb300 as idx
from paged_fp8_mqa_gb300 import synth
from gpu_cases import REL, ABS, expected_row_ends, to_device

pytestmark = pytest.mark.gpu


def test_withheld_tile_times_out_and_recovers():
    w = synth.make_workload("timeout", 71, 4, 1, 2048, "fixed", values=[2048, 1000, 512, 1500])
    t = to_device(w)
    pad = idx.idx_padded_seq_len(w.max_seq_len)
    ref, tol = oracle.paged_logits(w.q, w.kv_fused, w.weights, w.block_tables, w.seq_lens,
                                   w.max_seq_len, block_size=w.block_size)
    sched = oracle.schedule(w.seq_lens, idx.TILE_TOKENS, 4)  # 4 CTAs: which tiles each owns
    idx.device_status(clear=True)
    out = torch.full((w.rows, pad), float("nan"), device=t["q"].device)
    idx.idx_debug_withhold_first_tile(1)
    try:
        idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len,
                       out=out, num_sms=4)
        torch.cuda.synchronize()  # returns: every wait is time-limited
    finally:
        idx.idx_debug_withhold_first_tile(-1)
    assert idx.device_status(clear=True) & idx.IDX_DEV_WAIT_TIMEOUT
    got = out.cpu().double().numpy()
    # CTA 1 gave up at its first tile; CTAs 0, 2 and 3 finished: their tiles match the oracle.
    tiles = []
    for b in range(w.batch):
        for j in range(-(-int(w.seq_lens[b]) // idx.TILE_TOKENS)):
            tiles.append((b, j))
    cta_of = {}
    starts = [tuple(x) for x in sched.tolist()]
    flat = {bt: i for i, bt in enumerate(tiles)}
    bounds = [flat.get(s, len(tiles)) for s in starts]
    for c in range(4):
        for f in range(bounds[c], bounds[c + 1]):
            cta_of[tiles[f]] = c
    re = expected_row_ends(w)
    checked = 0
    for (b, j), c in cta_of.items():
        if c == 1:
            continue
        lo, hi = j * idx.TILE_TOKENS, min((j + 1) * idx.TILE_TOKENS, int(re[b]))
        err = np.abs(got[b, lo:hi] - ref[b, lo:hi])
        assert (err <= REL * tol[b, lo:hi] + ABS).all(), (b, j)
        checked += hi - lo
    assert checked > 0
    # The context is usable and the next launch (injection off) is complete and correct.
    out.fill_(float("nan"))
    idx.logits_fp8(t["q"], t["kv"], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len,
                   out=out, num_sms=4)
    torch.cuda.synchronize()
    assert idx.device_status(clear=True) == 0
    got = out.cpu().double().numpy()
    for r in range(w.rows):
        e = int(re[r])
        assert (np.abs(got[r, :e] - ref[r, :e]) <= REL * tol[r, :e] + ABS).all()


def test_injection_argument_checked():
    with pytest.raises(idx.IdxError):
        idx.idx_debug_withhold_first_tile(-2)
    with pytest.raises(idx.IdxError):
        idx.idx_debug_withhold_first_tile(1024)
