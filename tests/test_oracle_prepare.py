"""Pins for the oracle's prepare_block (CPU only).

"From DFlash to dLLM Self-Spec (II)", section 2.2.2: slot 0 of each block holds
the last verified token and the other slots hold the mask token; the block's
positions continue the committed sequence and its cache slots come from the
request's page mapping.  Pinned here by a round trip through a paged pool: a
value written at logical position t of request r (through the block table) is
read back at cache_loc of the slot whose position is t.
"""
import numpy as np

import oracle
from block_diffusion_speculative_attn_gb300 import workloads as wl


def test_block_layout_and_round_trip():
    rng = np.random.default_rng(3)
    for ps in (1, 4, 16, 64):
        seq_lens = rng.integers(0, 300, 9).astype(np.int32)
        B = 7
        table, num_pages = wl.paging_for(seq_lens, B, ps, rng, extra_pages=5)
        verified = rng.integers(0, 1000, len(seq_lens)).astype(np.int32)
        ids, pos, loc, bad = oracle.prepare_block(verified, seq_lens, table, num_pages, B, ps, 999)
        assert bad == 0
        assert (ids[:, 0] == verified).all() and (ids[:, 1:] == 999).all()
        # write "request*10^6 + position" at every logical position through the table
        pool = np.full(num_pages * ps, -1, np.int64)
        for r, L in enumerate(seq_lens):
            for t in range(L + B):
                pool[table[r, t // ps] * ps + t % ps] = r * 10**6 + t
        for r, L in enumerate(seq_lens):
            assert pos[r].tolist() == list(range(L, L + B))
            assert pool[loc[r]].tolist() == [r * 10**6 + t for t in range(L, L + B)]


def test_out_of_range_is_counted():
    seq_lens = np.asarray([6, 3], np.int32)
    table = np.asarray([[0, 1, 2], [3, 99, -1]], np.int32)
    ids, pos, loc, bad = oracle.prepare_block(np.asarray([1, 2], np.int32), seq_lens, table, 4,
                                              4, 4, 0)
    # request 1 needs pages 0 and 1 of its table; page id 99 is outside the pool of 4
    assert bad == 3 and (loc[1, 1:] == -1).all() and loc[1, 0] == 3 * 4 + 3
    assert (loc[0] >= 0).all()
