"""Pins for the oracle's speculative acceptance (CPU only).

Rules pinned (oracle/bdsa_oracle.c, oracle_spec_accept):
* hand-worked cases under tests/golden/accept_cases.json, each citing the rule
  it applies ("From DFlash to dLLM Self-Spec (IV)", section 4.3.1 and the
  section 4.4.1 loop; "... (II)", section 2.2.5; "Unlocking Lossless Speedups
  in LLMs via Discrete Diffusion", background on speculative decoding);
* the sampling rule against numpy's cumsum + searchsorted;
* losslessness, the defining property of the rule on the Uno page: emitted
  tokens follow the verifier distribution (chi-square over 10^6 rows), and
  the first draft is accepted with probability sum_x min(p, q) = 1 - TV(p, q)
  (Leviathan et al., corollary 3.6, which the Uno page cites for its TV loss);
* q == p accepts everything; a one-hot verifier forces the token; the
  tokens-per-forward bound 1 <= commit_len <= B.
"""
import json
import os

import numpy as np
import pytest
from scipy import stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_cases.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_golden_cases(case):
    B, V = case["B"], case["V"]
    p = np.asarray(case["p"], np.float32)[None]
    q = None if case.get("greedy") else np.asarray(case["q"], np.float32)[None]
    out = oracle.spec_accept(np.asarray([case["block_ids"]], np.int32), p, q,
                             np.asarray([case["u_acc"]], np.float32),
                             np.asarray([case["u_samp"]], np.float32),
                             np.asarray([case["seq_len"]], np.int32))
    e = case["expect"]
    assert out["accept_len"][0] == e["accept_len"]
    assert out["commit_len"][0] == e["commit_len"]
    assert out["out_tokens"][0].tolist() == e["out_tokens"]
    assert out["bonus_id"][0] == e["bonus_id"]
    assert out["new_seq_lens"][0] == e["new_seq_len"]


def test_inv_cdf_matches_searchsorted():
    rng = np.random.default_rng(5)
    for trial in range(200):
        V = int(rng.integers(1, 300))
        w = rng.random(V).astype(np.float32)
        w[rng.random(V) < 0.3] = 0.0
        if not w.any():
            w[-1] = 1.0
        u = float(np.float32(rng.random()))
        c = np.cumsum(w.astype(np.float64))
        want = int(np.searchsorted(c, u * c[-1], side="right"))
        k, _ = oracle.inv_cdf(w, u)
        assert k == want
        assert w[k] > 0


def _sample(qrow: np.ndarray, u: np.ndarray) -> np.ndarray:
    c = np.cumsum(qrow.astype(np.float64))
    return np.minimum(np.searchsorted(c, u * c[-1], side="right"), len(qrow) - 1).astype(np.int32)


def _softmax(x):
    x = x - x.max(-1, keepdims=True)
    e = np.exp(x)
    return e / e.sum(-1, keepdims=True)


def _chisq_pvalue(counts: np.ndarray, probs: np.ndarray) -> float:
    n = counts.sum()
    exp = probs * n
    order = np.argsort(exp)
    oc, ec = [], []
    acc_o = acc_e = 0.0
    for k in order:  # merge the smallest-expectation bins until each has >= 5
        acc_o += counts[k]
        acc_e += exp[k]
        if acc_e >= 5.0:
            oc.append(acc_o)
            ec.append(acc_e)
            acc_o = acc_e = 0.0
    if acc_e > 0 and ec:
        oc[-1] += acc_o
        ec[-1] += acc_e
    oc, ec = np.asarray(oc), np.asarray(ec)
    stat = ((oc - ec) ** 2 / ec).sum()
    return float(stats.chi2.sf(stat, len(ec) - 1))


@pytest.fixture(scope="module")
def lossless_run():
    """10^6 rows, B = 8, V = 1000, p and q broadcast across rows (stride 0)."""
    rng = np.random.default_rng(2024)
    n, B, V = 1_000_000, 8, 1000
    p = _softmax(2.0 * rng.standard_normal((B, V))).astype(np.float32)
    q = _softmax(2.0 * rng.standard_normal((B - 1, V))).astype(np.float32)
    block_ids = np.empty((n, B), np.int32)
    block_ids[:, 0] = rng.integers(0, V, n)
    for i in range(1, B):
        block_ids[:, i] = _sample(q[i - 1], rng.random(n))
    u_acc = rng.random((n, B - 1), dtype=np.float32)
    u_samp = rng.random(n, dtype=np.float32)
    out = oracle.spec_accept(block_ids, p, q, u_acc, u_samp, np.zeros(n, np.int32),
                             p_strides=(0, V), q_strides=(0, V), V=V,
                             nthreads=max(1, os.cpu_count() or 1))
    return dict(p=p, q=q, out=out, n=n, B=B, V=V)


def test_lossless_chi_square(lossless_run):
    r = lossless_run
    a, toks = r["out"]["accept_len"], r["out"]["out_tokens"]
    for k in range(r["B"]):
        rows = a >= k
        if rows.sum() < 2000:
            continue
        counts = np.bincount(toks[rows, k], minlength=r["V"]).astype(np.float64)
        pv = _chisq_pvalue(counts, r["p"][k].astype(np.float64))
        assert pv > 1e-3, f"slot {k}: chi-square p-value {pv:.2e}"


def test_acceptance_rate_is_one_minus_tv(lossless_run):
    r = lossless_run
    a = r["out"]["accept_len"]
    for k in range(r["B"] - 1):
        reach = a >= k
        n = int(reach.sum())
        if n < 2000:
            continue
        emp = float((a[reach] >= k + 1).mean())
        want = float(np.minimum(r["p"][k].astype(np.float64), r["q"][k].astype(np.float64)).sum())
        sigma = np.sqrt(want * (1 - want) / n)
        assert abs(emp - want) < 5 * sigma + 1e-9, (k, emp, want, sigma)


def test_tokens_per_forward_bound(lossless_run):
    c = lossless_run["out"]["commit_len"]
    assert c.min() >= 1 and c.max() <= lossless_run["B"]
    assert (lossless_run["out"]["new_seq_lens"] == c).all()


def test_q_equal_p_accepts_all():
    rng = np.random.default_rng(6)
    bs, B, V = 64, 6, 50
    p = _softmax(rng.standard_normal((bs, B, V)) * 2).astype(np.float32)
    q = p[:, :B - 1].copy()
    ids = rng.integers(0, V, (bs, B)).astype(np.int32)
    u_samp = rng.random(bs, dtype=np.float32)
    out = oracle.spec_accept(ids, p, q, rng.random((bs, B - 1), dtype=np.float32), u_samp,
                             np.full(bs, 7, np.int32))
    assert (out["accept_len"] == B - 1).all()
    for r in range(bs):
        c = np.cumsum(p[r, B - 1].astype(np.float64))
        assert out["bonus_id"][r] == np.searchsorted(c, u_samp[r] * c[-1], side="right")
        assert out["out_tokens"][r, :B - 1].tolist() == ids[r, 1:].tolist()


def test_one_hot_verifier_forces_token():
    rng = np.random.default_rng(7)
    bs, B, V = 32, 5, 40
    hot = rng.integers(0, V, (bs, B))
    p = np.zeros((bs, B, V), np.float32)
    for r in range(bs):
        for i in range(B):
            p[r, i, hot[r, i]] = 1.0
    q = _softmax(rng.standard_normal((bs, B - 1, V))).astype(np.float32)
    ids = rng.integers(0, V, (bs, B)).astype(np.int32)
    out = oracle.spec_accept(ids, p, q, rng.random((bs, B - 1), dtype=np.float32),
                             rng.random(bs, dtype=np.float32), np.zeros(bs, np.int32))
    for r in range(bs):
        a = out["accept_len"][r]
        assert out["bonus_id"][r] == hot[r, a]
        for i in range(a):  # accepted drafts had verifier mass, i.e. were the hot token
            assert ids[r, i + 1] == hot[r, i]


def test_greedy_matches_argmax_prefix():
    rng = np.random.default_rng(8)
    bs, B, V = 200, 6, 30
    p = _softmax(3 * rng.standard_normal((bs, B, V))).astype(np.float32)
    am = p.argmax(-1)
    ids = rng.integers(0, V, (bs, B)).astype(np.int32)
    keep = rng.integers(0, B, bs)  # force a known matching prefix length
    for r in range(bs):
        ids[r, 1:1 + keep[r]] = am[r, :keep[r]]
    out = oracle.spec_accept(ids, p, None, np.zeros((bs, B - 1), np.float32),
                             np.zeros(bs, np.float32), np.zeros(bs, np.int32))
    for r in range(bs):
        a = 0
        while a < B - 1 and ids[r, a + 1] == am[r, a]:
            a += 1
        assert out["accept_len"][r] == a >= min(keep[r], B - 1)
        assert out["bonus_id"][r] == am[r, a]
