"""Pins of the oracle's I-DLM Block-N round ("From DFlash to dLLM Self-Spec (IV)",
sections 4.3, 4.3.1 and 4.6) against things other than itself:

* hand-worked rounds under tests/golden/idlm_cases.json, each citing its rule;
* the layout: slot 0 the pending token, the carried specs in slots 1..N-1 in
  verify mode, masks elsewhere, and cache locations equal to those of the
  (separately pinned) prepare_block for a block of 2N-1 slots;
* the draws of a cold start and of the new specs against numpy searchsorted
  on the cumulative weights;
* losslessness: with specs drawn from q, the first emitted token follows p[0],
  the second (given the first spec passed) p[1], and the bonus p[N-1], by
  chi-square; the first spec passes with probability sum min(p, q) = 1 - TV;
* q = p passes every spec; the verify outcome agrees with the pinned DFlash
  acceptance oracle on the same p / q rows; kv_keep = n_out = a + 1.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "idlm_cases.json")


def _cases():
    with open(GOLDEN) as fh:
        return json.load(fh)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_golden_rounds(case):
    N, V = case["N"], case["V"]
    blk = 2 * N - 1
    p = np.array(case["p"], np.float32).reshape(1, blk, V)
    q = np.array(case["q_prev"], np.float32).reshape(1, blk, V)
    ids = np.array(case["block_ids"], np.int32).reshape(1, blk)
    u_acc = np.array(case["u_acc"], np.float32).reshape(1, max(N - 1, 0))
    u_samp = np.array(case["u_samp"], np.float32).reshape(1, N)
    r = oracle.idlm_accept(ids, [case["mode"]], p, q, [case["q_slot"]], u_acc, u_samp,
                           [case["seq_len"]], N)
    e = case["expected"]
    assert r["accept_len"][0] == e["accept_len"]
    assert r["n_out"][0] == e["n_out"]
    assert r["out_tokens"][0].tolist() == e["out_tokens"]
    assert r["next_mode"][0] == e["next_mode"]
    assert r["next_pending"][0] == e["next_pending"]
    assert r["next_specs"][0].tolist() == e["next_specs"]
    assert r["next_q_slot"][0] == e["next_q_slot"]
    assert r["new_seq_lens"][0] == e["new_seq_len"]
    assert r["kv_keep"][0] == e["kv_keep"]


def _table(rng, bs, max_pages, num_pages):
    return rng.permutation(num_pages)[: bs * max_pages].reshape(bs, max_pages).astype(np.int32)


@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_layout_and_cache_locations(N):
    rng = np.random.default_rng(5 + N)
    bs, ps, mask = 6, 8, 99
    blk = 2 * N - 1
    seq = rng.integers(0, 60, bs).astype(np.int32)
    max_pages = (60 + blk) // ps + 1
    table = _table(rng, bs, max_pages, bs * max_pages + 3)
    pending = rng.integers(0, 50, bs).astype(np.int32)
    specs = rng.integers(0, 50, (bs, max(N - 1, 0))).astype(np.int32)
    mode = np.array([1, 0, 1, 1, 0, 1], np.int32)
    ids, pos, loc, bad = oracle.idlm_prepare(pending, specs, mode, seq, table,
                                             table.size + 3, N, ps, mask)
    assert bad == 0
    for r in range(bs):
        assert ids[r, 0] == pending[r]
        if mode[r] == 1:
            assert ids[r, 1:N].tolist() == specs[r].tolist()
            assert (ids[r, N:] == mask).all()
        else:
            assert (ids[r, 1:] == mask).all()
        assert pos[r].tolist() == list(range(seq[r], seq[r] + blk))
    _, _, loc_ref, _ = oracle.prepare_block(pending, seq, table, table.size + 3, blk, ps, mask)
    np.testing.assert_array_equal(loc, loc_ref)


def _softmax(x):
    e = np.exp(x - x.max(-1, keepdims=True))
    return (e / e.sum(-1, keepdims=True)).astype(np.float32)


def _draw(w, u):
    c = np.cumsum(np.asarray(w, np.float64))
    return int(np.searchsorted(c, u * c[-1], side="right"))


def test_cold_start_and_new_specs_match_searchsorted():
    rng = np.random.default_rng(11)
    bs, N, V = 64, 5, 50
    blk = 2 * N - 1
    p = _softmax(rng.normal(0, 2, (bs, blk, V)))
    ids = np.full((bs, blk), 7, np.int32)
    u_samp = rng.random((bs, N), dtype=np.float32)
    r = oracle.idlm_accept(ids, np.zeros(bs, np.int32), p, p, np.ones(bs, np.int32),
                           np.zeros((bs, N - 1), np.float32), u_samp, np.zeros(bs, np.int32), N)
    keep = r["flags"] == 0
    assert keep.mean() > 0.9
    for i in np.nonzero(keep)[0]:
        assert r["next_pending"][i] == _draw(p[i, 0], u_samp[i, 0])
        for j in range(N - 1):
            assert r["next_specs"][i, j] == _draw(p[i, 1 + j], u_samp[i, 1 + j])
    assert (r["next_q_slot"] == 1).all() and (r["next_mode"] == 1).all()
    assert (r["kv_keep"] == 1).all() and (r["n_out"] == 1).all()


@pytest.fixture(scope="module")
def lossless_run():
    """Many independent rounds in verify mode on one small distribution set:
    specs drawn from their q rows, fresh uniforms per row."""
    rng = np.random.default_rng(2024)
    n, N, V = 400_000, 4, 6
    blk = 2 * N - 1
    p1 = _softmax(rng.normal(0, 1.5, (blk, V)))
    q1 = _softmax(rng.normal(0, 1.5, (blk, V)))
    q_slot = 2
    qw = q1.astype(np.float64)
    specs = np.stack([rng.choice(V, n, p=qw[q_slot + k] / qw[q_slot + k].sum())
                      for k in range(N - 1)], 1)
    ids = np.full((n, blk), V + 1, np.int32)
    ids[:, 0] = 0
    ids[:, 1:N] = specs
    u_acc = rng.random((n, N - 1), dtype=np.float32)
    u_samp = rng.random((n, N), dtype=np.float32)
    r = oracle.idlm_accept(ids, np.ones(n, np.int32), p1[None], q1[None],
                           np.full(n, q_slot, np.int32), u_acc, u_samp, np.zeros(n, np.int32), N,
                           p_strides=(0, V), q_strides=(0, V), V=V,
                           nthreads=oracle.max_threads())
    return p1, q1, q_slot, N, V, r


def _chi2_ok(counts, probs):
    from scipy import stats
    n = counts.sum()
    exp = probs / probs.sum() * n
    keep = exp >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    ex = np.append(exp[keep], exp[~keep].sum())
    if ex[-1] == 0:
        obs, ex = obs[:-1], ex[:-1]
    stat = ((obs - ex) ** 2 / ex).sum()
    return stats.chi2.sf(stat, len(obs) - 1) > 1e-3


def test_lossless_first_second_and_bonus(lossless_run):
    p1, q1, q_slot, N, V, r = lossless_run
    out, a = r["out_tokens"], r["accept_len"]
    assert _chi2_ok(np.bincount(out[:, 0], minlength=V), p1[0].astype(np.float64))
    sel = a >= 1
    assert _chi2_ok(np.bincount(out[sel, 1], minlength=V), p1[1].astype(np.float64))
    full = a == N - 1
    assert full.sum() > 1000
    assert _chi2_ok(np.bincount(out[full, N - 1], minlength=V), p1[N - 1].astype(np.float64))
    for j in range(N - 1):
        assert _chi2_ok(np.bincount(r["next_specs"][full, j], minlength=V),
                        p1[N + j].astype(np.float64))


def test_first_spec_acceptance_rate(lossless_run):
    p1, q1, q_slot, N, V, r = lossless_run
    n = len(r["accept_len"])
    rate = (r["accept_len"] >= 1).mean()
    expect = np.minimum(p1[0].astype(np.float64), q1[q_slot].astype(np.float64)).sum()
    assert abs(rate - expect) < 5 * np.sqrt(expect * (1 - expect) / n)


def test_round_invariants(lossless_run):
    p1, q1, q_slot, N, V, r = lossless_run
    a = r["accept_len"]
    assert ((a >= 0) & (a <= N - 1)).all()
    np.testing.assert_array_equal(r["n_out"], a + 1)
    np.testing.assert_array_equal(r["kv_keep"], a + 1)
    np.testing.assert_array_equal(r["new_seq_lens"], a + 1)
    rows = np.arange(len(a))
    np.testing.assert_array_equal(r["next_pending"], r["out_tokens"][rows, a])
    full = a == N - 1
    assert (r["next_mode"][full] == 1).all() and (r["next_q_slot"][full] == N).all()
    assert (r["next_mode"][~full] == 0).all() and (r["next_specs"][~full] == -1).all()


def test_q_equal_p_passes_every_spec():
    rng = np.random.default_rng(3)
    bs, N, V = 200, 6, 30
    blk = 2 * N - 1
    p = _softmax(rng.normal(0, 2, (bs, blk, V)))
    q_prev = np.zeros_like(p)
    q_prev[:, 1:N] = p[:, 0:N - 1]  # q_slot = 1: spec_k's q row equals p[k]
    ids = np.zeros((bs, blk), np.int32)
    for i in range(bs):
        for k in range(N - 1):
            w = p[i, k].astype(np.float64)
            ids[i, 1 + k] = rng.choice(V, p=w / w.sum())
    r = oracle.idlm_accept(ids, np.ones(bs, np.int32), p, q_prev, np.ones(bs, np.int32),
                           rng.random((bs, N - 1), dtype=np.float32),
                           rng.random((bs, N), dtype=np.float32), np.zeros(bs, np.int32), N)
    assert (r["accept_len"] == N - 1).all()


def test_verify_agrees_with_block_acceptance():
    """A verify round is DFlash acceptance over the block [pending, specs]
    with p rows 0..N-1 and q rows q_slot..q_slot+N-2 (same uniforms)."""
    rng = np.random.default_rng(8)
    bs, N, V = 300, 5, 40
    blk = 2 * N - 1
    p = _softmax(rng.normal(0, 2, (bs, blk, V)))
    q_prev = _softmax(rng.normal(0, 2, (bs, blk, V)))
    q_slot = rng.integers(0, N + 1, bs).astype(np.int32)
    ids = rng.integers(0, V, (bs, blk)).astype(np.int32)
    u_acc = rng.random((bs, N - 1), dtype=np.float32)
    u_samp = rng.random((bs, N), dtype=np.float32)
    r = oracle.idlm_accept(ids, np.ones(bs, np.int32), p, q_prev, q_slot, u_acc, u_samp,
                           np.full(bs, 10, np.int32), N)
    q_rows = np.stack([q_prev[i, q_slot[i]:q_slot[i] + N - 1] for i in range(bs)])
    ref = oracle.spec_accept(ids[:, :N], p[:, :N], q_rows, u_acc, u_samp[:, 0],
                             np.full(bs, 10, np.int32))
    np.testing.assert_array_equal(r["accept_len"], ref["accept_len"])
    np.testing.assert_array_equal(r["out_tokens"], ref["out_tokens"])
    np.testing.assert_array_equal(r["new_seq_lens"], ref["new_seq_lens"])


def test_bad_q_slot_and_mode_fall_back_to_cold_start():
    rng = np.random.default_rng(9)
    N, V = 3, 10
    blk = 2 * N - 1
    p = _softmax(rng.normal(0, 2, (3, blk, V)))
    ids = np.zeros((3, blk), np.int32)
    u_samp = rng.random((3, N), dtype=np.float32)
    r = oracle.idlm_accept(ids, np.array([1, 5, 0], np.int32), p, p,
                           np.array([N + 1, 1, 1], np.int32), np.zeros((3, N - 1), np.float32),
                           u_samp, np.zeros(3, np.int32), N)
    assert r["flags"][0] & 32 and r["flags"][1] & 64
    ref = oracle.idlm_accept(ids, np.zeros(3, np.int32), p, p, np.ones(3, np.int32),
                             np.zeros((3, N - 1), np.float32), u_samp, np.zeros(3, np.int32), N)
    for k in ("next_pending", "next_specs", "kv_keep", "next_q_slot"):
        np.testing.assert_array_equal(r[k], ref[k])
