"""Pins of oracle.append_block_kv (the block's own K/V written into the paged
cache, "From DFlash to dLLM Self-Spec (II)", sections 2.2.2 and 2.2.4).

The written rows must be exactly the cache locations that the C oracle's
prepare_block computes for the block's positions (an independent definition),
nothing else may change, rows on pages outside the pool are skipped, and an
append of rows already in the cache leaves the attention unchanged.
"""
import numpy as np

import oracle
from block_diffusion_speculative_attn_gb300 import workloads as wl


def _case(seed=5, bs=3, B=8, Hkv=2, D=16, ps=16, lens=(40, 0, 77)):
    rng = np.random.default_rng(seed)
    bt, num_pages = wl.paging_for(np.array(lens, np.int32), B, ps, rng)
    slots = num_pages * ps
    k = rng.integers(0, 1 << 16, (slots, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, (slots, Hkv, D), dtype=np.uint16)
    kn = rng.integers(0, 1 << 16, (bs * B, Hkv, D), dtype=np.uint16)
    vn = rng.integers(0, 1 << 16, (bs * B, Hkv, D), dtype=np.uint16)
    return np.array(lens, np.int32), bt, num_pages, k, v, kn, vn


def test_writes_exactly_the_prepare_block_cache_locations():
    sl, bt, num_pages, k, v, kn, vn = _case()
    B, ps = 8, 16
    k2, v2 = oracle.append_block_kv(k, v, kn, vn, bt, sl, B, ps, num_pages)
    _, _, cache_loc, bad = oracle.prepare_block(np.zeros(len(sl), np.int32), sl, bt, num_pages, B,
                                                ps, 0)
    assert bad == 0
    loc = cache_loc.reshape(-1)
    assert len(set(loc.tolist())) == loc.size  # distinct slots
    np.testing.assert_array_equal(k2[loc], kn)
    np.testing.assert_array_equal(v2[loc], vn)
    keep = np.ones(k.shape[0], bool)
    keep[loc] = False
    np.testing.assert_array_equal(k2[keep], k[keep])
    np.testing.assert_array_equal(v2[keep], v[keep])
    # the inputs are not modified
    assert not np.array_equal(k2, k)


def test_pages_outside_the_pool_are_not_written():
    sl, bt, num_pages, k, v, kn, vn = _case()
    B, ps = 8, 16
    bt = bt.copy()
    page = int(sl[0]) // ps
    bt[0, page] = num_pages + 3           # request 0's block page is outside the pool
    k2, v2 = oracle.append_block_kv(k, v, kn, vn, bt, sl, B, ps, num_pages)
    _, _, cache_loc, bad = oracle.prepare_block(np.zeros(len(sl), np.int32), sl, bt, num_pages, B,
                                                ps, 0)
    assert bad > 0
    # request 0's rows on the bad page are skipped; every other written row matches
    for r in range(len(sl)):
        for i in range(B):
            c = int(cache_loc[r, i])
            if c < 0:
                continue
            np.testing.assert_array_equal(k2[c], kn[r * B + i])
    written = {int(c) for c in cache_loc.reshape(-1) if c >= 0}
    keep = np.array([s not in written for s in range(k.shape[0])])
    np.testing.assert_array_equal(k2[keep], k[keep])


def test_negative_length_writes_nothing():
    sl, bt, num_pages, k, v, kn, vn = _case(lens=(40, 0, 77))
    sl = sl.copy()
    sl[1] = -1
    k2, _ = oracle.append_block_kv(k, v, kn, vn, bt, sl, 8, 16, num_pages)
    sl2 = sl.copy()
    k3, _ = oracle.append_block_kv(k, v, kn, vn, bt, np.where(sl2 < 0, 0, sl2), 8, 16, num_pages)
    # request 1 writes nothing with L = -1, but writes its rows with L = 0
    assert not np.array_equal(k2, k3)
    rows1 = [int(bt[1, 0]) * 16 + i for i in range(8)]
    np.testing.assert_array_equal(k2[rows1], k[rows1])


def test_reappending_cached_rows_changes_nothing():
    # make_attn_inputs already holds the block's K/V in the cache; appending those
    # same rows must leave the caches, and so the attention, unchanged
    cfg = wl.config("tiny")
    inp = wl.make_attn_inputs(cfg)
    kb, vb = wl.bf16_bits(inp.k_cache), wl.bf16_bits(inp.v_cache)
    _, _, cache_loc, bad = oracle.prepare_block(np.zeros(cfg.bs, np.int32), inp.seq_lens,
                                                inp.block_table, inp.num_pages, cfg.B,
                                                cfg.page_size, 0)
    loc = cache_loc.reshape(-1)
    k2, v2 = oracle.append_block_kv(kb, vb, kb[loc], vb[loc], inp.block_table, inp.seq_lens,
                                    cfg.B, cfg.page_size, inp.num_pages)
    np.testing.assert_array_equal(k2, kb)
    np.testing.assert_array_equal(v2, vb)
