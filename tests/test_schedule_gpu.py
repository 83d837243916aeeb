"""The standalone schedule kernel against the oracle's work split, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import paged_fp8_mqa_gb300 as idx

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(6))
def test_schedule_matches_oracle(seed):
    g = torch.Generator().manual_seed(seed)
    B = int(torch.randint(1, 4097 if seed == 5 else 300, (1,), generator=g))
    lens = torch.randint(0, 70000, (B,), generator=g).to(torch.int32)
    lens[torch.rand(B, generator=g) < 0.15] = 0
    for n_sms in (1, 7, 152, 1024):
        got = idx.schedule(lens.cuda(), 1, n_sms).cpu().numpy()
        ref = oracle.schedule(lens, idx.TILE_TOKENS, n_sms)
        assert (got == ref).all(), (B, n_sms)


def test_schedule_strided_lengths():
    lens = torch.tensor([100, -1, 5000, -1, 0, -1, 129, -1], dtype=torch.int32).cuda()
    got = idx.schedule(lens[::2], 2, 5).cpu().numpy()
    ref = oracle.schedule(lens[::2].cpu(), idx.TILE_TOKENS, 5)
    assert (got == ref).all()
