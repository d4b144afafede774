"""GPU parity of bdsa_prepare_block against the oracle (bit-exact integers)."""
import numpy as np
import pytest
import torch

import block_diffusion_speculative_attn_gb300 as bdsa
import oracle
from block_diffusion_speculative_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ps", [1, 8, 16, 64, 1024])
@pytest.mark.parametrize("B", [1, 8, 16, 64])
def test_matches_oracle(ps, B):
    rng = np.random.default_rng(ps * 7 + B)
    bs = 300
    seq_lens = rng.integers(0, 5000, bs).astype(np.int32)
    table, num_pages = wl.paging_for(seq_lens, B, ps, rng, extra_pages=3)
    verified = rng.integers(0, 151936, bs).astype(np.int32)
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    got = bdsa.prepare_block(torch.from_numpy(verified).to(dev), torch.from_numpy(seq_lens).to(dev),
                             torch.from_numpy(table).to(dev), num_pages, B, ps, 151665,
                             dev_status=status)
    want = oracle.prepare_block(verified, seq_lens, table, num_pages, B, ps, 151665)
    for g, w in zip(got, want[:3]):
        assert (g.cpu().numpy() == w).all()
    assert status.item() == 0 and want[3] == 0


def test_out_of_range_flags_and_marks():
    dev = torch.device("cuda")
    seq_lens = np.asarray([6, 3], np.int32)
    table = np.asarray([[0, 1, 2], [3, 99, -1]], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ids, pos, loc = bdsa.prepare_block(torch.tensor([1, 2], dtype=torch.int32, device=dev),
                                       torch.from_numpy(seq_lens).to(dev),
                                       torch.from_numpy(table).to(dev), 4, 4, 4, 0,
                                       dev_status=status)
    want = oracle.prepare_block(np.asarray([1, 2], np.int32), seq_lens, table, 4, 4, 4, 0)
    assert (loc.cpu().numpy() == want[2]).all()
    assert status.item() == 16
