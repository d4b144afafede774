"""GPU parity of the I-DLM Block-N round ("From DFlash to dLLM Self-Spec (IV)",
sections 4.3, 4.3.1 and 4.6): bdsa_idlm_prepare and bdsa_idlm_accept against
the fp64 oracle.

Everything is integer output, so the bar is bit-exact.  The acceptance test is
the same IEEE fp32 divide and compare on both sides; a draw compares u*S with
cumulative sums, and rows where the oracle finds u*S within 1e-9*S of the
chosen token's boundary (flag bit 1, any of the row's draws) are excluded and
counted, as in the DFlash acceptance tests.
"""
import json
import os

import numpy as np
import pytest
import torch

import block_diffusion_speculative_attn_gb300 as bdsa
import oracle
from block_diffusion_speculative_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
KEYS = bdsa.IDLM_KEYS + ("out_tokens", "next_specs")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "idlm_cases.json")
DEV = "cuda"


def _t(x, dtype):
    return torch.as_tensor(np.ascontiguousarray(x), dtype=dtype, device=DEV)


def _softmax(x):
    e = np.exp(x - x.max(-1, keepdims=True))
    return (e / e.sum(-1, keepdims=True)).astype(np.float32)


def _compare(got, want, max_flag_frac=1e-3):
    ok = (want["flags"] & 2) == 0
    assert (~ok).mean() <= max_flag_frac, f"{(~ok).sum()} flagged rows"
    for k in KEYS:
        g = got[k].cpu().numpy()
        w = want[k]
        if w.size == 0:
            assert g.size == 0, k
            continue
        bad = (g != w).reshape(len(ok), -1).any(-1) & ok
        assert not bad.any(), (k, np.nonzero(bad)[0][:10], g[bad][:3], w[bad][:3])
    return int((~ok).sum())


def _gpu_accept(ids, mode, p, q, q_slot, u_acc, u_samp, seq, N, status=None, sms=0, **kw):
    return bdsa.idlm_accept(_t(ids, torch.int32), _t(mode, torch.int32), _t(p, torch.float32),
                            _t(q, torch.float32), _t(q_slot, torch.int32),
                            _t(u_acc, torch.float32), _t(u_samp, torch.float32),
                            _t(seq, torch.int32), N, dev_status=status, sms=sms, **kw)


# ------------------------------------------------------------------ prepare
@pytest.mark.parametrize("ps", [1, 16, 64])
@pytest.mark.parametrize("N", [1, 2, 8, 16])
def test_prepare_matches_oracle(N, ps):
    rng = np.random.default_rng(N * 31 + ps)
    bs, blk, mask = 257, 2 * N - 1, 151665
    seq = rng.integers(0, 5000, bs).astype(np.int32)
    table, num_pages = wl.paging_for(seq, blk, ps, rng, extra_pages=3)
    pending = rng.integers(0, 151936, bs).astype(np.int32)
    specs = rng.integers(0, 151936, (bs, max(N - 1, 0))).astype(np.int32)
    mode = rng.integers(0, 2, bs).astype(np.int32)
    mode[:3] = (7, -1, 1)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = bdsa.idlm_prepare(_t(pending, torch.int32), _t(specs, torch.int32),
                            _t(mode, torch.int32), _t(seq, torch.int32), _t(table, torch.int32),
                            num_pages, N, ps, mask, dev_status=status)
    want = oracle.idlm_prepare(pending, specs, mode, seq, table, num_pages, N, ps, mask)
    for g, w in zip(got, want[:3]):
        np.testing.assert_array_equal(g.cpu().numpy(), w)
    assert want[3] == 0 and status.item() == 0


def test_prepare_out_of_range_marks_and_flags():
    N, ps = 3, 4
    seq = np.asarray([2, 3, -1], np.int32)
    table = np.asarray([[0, 1, 2], [3, 99, -1], [4, 5, 6]], np.int32)
    pending = np.asarray([1, 2, 3], np.int32)
    specs = np.asarray([[5, 6], [7, 8], [9, 10]], np.int32)
    mode = np.asarray([1, 1, 0], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = bdsa.idlm_prepare(_t(pending, torch.int32), _t(specs, torch.int32),
                            _t(mode, torch.int32), _t(seq, torch.int32), _t(table, torch.int32),
                            7, N, ps, 0, dev_status=status)
    want = oracle.idlm_prepare(pending, specs, mode, seq, table, 7, N, ps, 0)
    for g, w in zip(got, want[:3]):
        np.testing.assert_array_equal(g.cpu().numpy(), w)
    assert want[3] > 0 and status.item() == 16


# ------------------------------------------------------------------- accept
@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_golden_rounds(case):
    N, V = case["N"], case["V"]
    blk = 2 * N - 1
    p = np.array(case["p"], np.float32).reshape(1, blk, V)
    q = np.array(case["q_prev"], np.float32).reshape(1, blk, V)
    ids = np.array(case["block_ids"], np.int32).reshape(1, blk)
    u_acc = np.array(case["u_acc"], np.float32).reshape(1, max(N - 1, 0))
    u_samp = np.array(case["u_samp"], np.float32).reshape(1, N)
    r = _gpu_accept(ids, [case["mode"]], p, q, [case["q_slot"]], u_acc, u_samp,
                    [case["seq_len"]], N)
    e = case["expected"]
    assert r["accept_len"].item() == e["accept_len"]
    assert r["n_out"].item() == e["n_out"]
    assert r["out_tokens"][0].tolist() == e["out_tokens"]
    assert r["next_mode"].item() == e["next_mode"]
    assert r["next_pending"].item() == e["next_pending"]
    assert r["next_specs"][0].tolist() == e["next_specs"]
    assert r["next_q_slot"].item() == e["next_q_slot"]
    assert r["new_seq_lens"].item() == e["new_seq_len"]
    assert r["kv_keep"].item() == e["kv_keep"]


def _random_round(rng, bs, N, V, alpha=0.3):
    """Dirichlet p / q_prev rows; verify rows carry specs drawn from their q rows."""
    blk = 2 * N - 1
    p = rng.dirichlet(np.full(V, alpha), (bs, blk)).astype(np.float32)
    q = rng.dirichlet(np.full(V, alpha), (bs, blk)).astype(np.float32)
    mode = (rng.random(bs) < 0.75).astype(np.int32)
    q_slot = rng.integers(0, N + 1, bs).astype(np.int32)
    ids = rng.integers(0, V, (bs, blk)).astype(np.int32)
    for k in range(N - 1):
        rows = q[np.arange(bs), q_slot + k]
        ids[:, 1 + k] = wl.draft_from(rows, rng.random(bs))
    u_acc = rng.random((bs, max(N - 1, 0)), dtype=np.float32)
    u_samp = rng.random((bs, N), dtype=np.float32)
    seq = rng.integers(0, 5000, bs).astype(np.int32)
    return ids, mode, p, q, q_slot, u_acc, u_samp, seq


@pytest.mark.parametrize("V", [1, 7, 256, 257, 4099])
@pytest.mark.parametrize("N", [1, 2, 3, 8, 32])
def test_ragged_vocab_and_block(N, V):
    rng = np.random.default_rng(N * 1000 + V)
    args = _random_round(rng, 48, N, V)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _gpu_accept(*args, N, status=status)
    want = oracle.idlm_accept(*args, N)
    _compare(got, want, max_flag_frac=0.05)
    assert status.item() == 0


@pytest.mark.parametrize("sms", [0, 1, 4096])
def test_chunking_does_not_change_results(sms):
    rng = np.random.default_rng(77)
    N, V = 4, 20000
    args = _random_round(rng, 40, N, V, alpha=1.0)
    got = _gpu_accept(*args, N, sms=sms)
    want = oracle.idlm_accept(*args, N)
    _compare(got, want, max_flag_frac=0.05)


def test_strided_broadcast_rows():
    """p and q_prev addressed through strides: one distribution set shared by
    every request (row stride 0), as a caller keeping one copy would."""
    rng = np.random.default_rng(5)
    bs, N, V = 4096, 4, 300
    blk = 2 * N - 1
    p1 = _softmax(rng.normal(0, 1.5, (blk, V)))
    q1 = _softmax(rng.normal(0, 1.5, (blk, V)))
    q_slot = np.full(bs, 2, np.int32)
    ids = np.zeros((bs, blk), np.int32)
    for k in range(N - 1):
        ids[:, 1 + k] = wl.draft_from(np.broadcast_to(q1[2 + k], (bs, V)), rng.random(bs))
    mode = np.ones(bs, np.int32)
    u_acc = rng.random((bs, N - 1), dtype=np.float32)
    u_samp = rng.random((bs, N), dtype=np.float32)
    seq = np.zeros(bs, np.int32)
    got = bdsa.idlm_accept(_t(ids, torch.int32), _t(mode, torch.int32), _t(p1, torch.float32),
                           _t(q1, torch.float32), _t(q_slot, torch.int32),
                           _t(u_acc, torch.float32), _t(u_samp, torch.float32),
                           _t(seq, torch.int32), N, p_strides=(0, V), q_strides=(0, V), V=V)
    want = oracle.idlm_accept(ids, mode, p1[None], q1[None], q_slot, u_acc, u_samp, seq, N,
                              p_strides=(0, V), q_strides=(0, V), V=V)
    _compare(got, want, max_flag_frac=0.01)


def test_bad_mode_and_q_slot_flag_and_cold_start():
    rng = np.random.default_rng(9)
    N, V = 3, 64
    ids, mode, p, q, q_slot, u_acc, u_samp, seq = _random_round(rng, 4, N, V)
    mode[:] = (1, 5, 0, 1)
    q_slot[:] = (N + 1, 1, 1, -1)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _gpu_accept(ids, mode, p, q, q_slot, u_acc, u_samp, seq, N, status=status)
    want = oracle.idlm_accept(ids, mode, p, q, q_slot, u_acc, u_samp, seq, N)
    _compare(got, want, max_flag_frac=0.5)
    assert status.item() == 16
    assert (got["next_q_slot"].cpu().numpy() == 1).all()


def test_spec_outside_vocab_rejects_and_flags():
    rng = np.random.default_rng(10)
    N, V = 4, 50
    ids, mode, p, q, q_slot, u_acc, u_samp, seq = _random_round(rng, 2, N, V)
    mode[:] = 1
    q_slot[:] = 1
    u_acc[:] = 0.0       # every in-vocabulary spec with p > 0 passes
    ids[0, 2] = V + 3    # spec_1 of row 0 is not a token
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _gpu_accept(ids, mode, p, q, q_slot, u_acc, u_samp, seq, N, status=status)
    want = oracle.idlm_accept(ids, mode, p, q, q_slot, u_acc, u_samp, seq, N)
    _compare(got, want, max_flag_frac=1.0)
    assert got["accept_len"][0].item() == 1 and status.item() == 16


def test_chained_rounds_match_oracle():
    """Three rounds: each round's next_pending / next_specs / next_mode /
    next_q_slot / new_seq_lens feed the next round's layout, and its p rows are
    the next round's q_prev.  GPU and oracle chains are run side by side."""
    rng = np.random.default_rng(21)
    bs, N, V, ps = 64, 5, 2000, 16
    blk = 2 * N - 1
    seq = rng.integers(0, 300, bs).astype(np.int32)
    table, num_pages = wl.paging_for(seq + 4 * blk, blk, ps, rng)
    pending = rng.integers(0, V, bs).astype(np.int32)
    specs = np.full((bs, N - 1), -1, np.int32)
    mode = np.zeros(bs, np.int32)
    q_slot = np.full(bs, -1, np.int32)
    q_prev = rng.dirichlet(np.full(V, 0.5), (bs, blk)).astype(np.float32)
    flagged = 0
    for _ in range(3):
        logits = rng.normal(0, 2, (bs, blk, V))
        p = _softmax(logits)
        # make the carried specs' verifier rows close to the rows they were drawn from
        for r in range(bs):
            if mode[r] == 1:
                p[r, :N - 1] = _softmax(np.log(q_prev[r, q_slot[r]:q_slot[r] + N - 1] + 1e-30)
                                        + rng.normal(0, 0.5, (N - 1, V)))
        ids_g, pos_g, loc_g = bdsa.idlm_prepare(
            _t(pending, torch.int32), _t(specs, torch.int32), _t(mode, torch.int32),
            _t(seq, torch.int32), _t(table, torch.int32), num_pages, N, ps, V - 1)
        ids, pos, loc, bad = oracle.idlm_prepare(pending, specs, mode, seq, table, num_pages, N,
                                                 ps, V - 1)
        assert bad == 0
        np.testing.assert_array_equal(ids_g.cpu().numpy(), ids)
        np.testing.assert_array_equal(loc_g.cpu().numpy(), loc)
        u_acc = rng.random((bs, N - 1), dtype=np.float32)
        u_samp = rng.random((bs, N), dtype=np.float32)
        got = bdsa.idlm_accept(ids_g, _t(mode, torch.int32), _t(p, torch.float32),
                               _t(q_prev, torch.float32), _t(q_slot, torch.int32),
                               _t(u_acc, torch.float32), _t(u_samp, torch.float32),
                               _t(seq, torch.int32), N)
        want = oracle.idlm_accept(ids, mode, p, q_prev, q_slot, u_acc, u_samp, seq, N)
        flagged += _compare(got, want, max_flag_frac=0.05)
        # carry the oracle's state so that both sides see identical next rounds
        pending, specs = want["next_pending"], want["next_specs"]
        mode, q_slot, seq = want["next_mode"], want["next_q_slot"], want["new_seq_lens"]
        q_prev = p
    assert flagged <= 3


@pytest.fixture(scope="module")
def qwen_round():
    cfg = wl.config("qwen3_8b_verify")
    return wl.make_idlm_inputs(cfg, N=8, device=DEV)


def test_qwen3_8b_shaped_round(qwen_round):
    """Batch 32, vocabulary 151936, N = 8 (15 slots), 3 in 4 requests verify:
    the full-size launch the benchmark times, every row compared."""
    x, N = qwen_round, qwen_round.N
    cfg = wl.config("qwen3_8b_verify")
    bs = x.pending.shape[0]
    rng = np.random.default_rng(3)
    seq = x.seq_lens.cpu().numpy()
    table, num_pages = wl.paging_for(seq, 2 * N - 1, cfg.page_size, rng)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids, _, _ = bdsa.idlm_prepare(x.pending, x.specs, x.mode, x.seq_lens,
                                  _t(table, torch.int32), num_pages, N, cfg.page_size,
                                  cfg.mask_token_id, dev_status=status)
    got = bdsa.idlm_accept(ids, x.mode, x.p, x.q_prev, x.q_slot, x.u_acc, x.u_samp,
                           x.seq_lens, N, dev_status=status)
    torch.cuda.synchronize()
    want = oracle.idlm_accept(ids.cpu().numpy(), x.mode.cpu().numpy(), x.p.cpu().numpy(),
                              x.q_prev.cpu().numpy(), x.q_slot.cpu().numpy(),
                              x.u_acc.cpu().numpy(), x.u_samp.cpu().numpy(), seq, N,
                              nthreads=oracle.max_threads())
    _compare(got, want, max_flag_frac=2 / bs)
    assert status.item() == 0
    a = got["accept_len"].cpu().numpy()
    verify = x.mode.cpu().numpy() == 1
    assert (a[~verify] == 0).all() and a[verify].max() > 0
