"""Pins of the oracle's tree verify ("Unlocking Lossless Speedups in LLMs via
Discrete Diffusion", Psi-Spec Tree sampler; "SGLang dLLM / LLaDA 2.0",
"Attention Mask") against things other than itself:

* hand-worked cases in tests/golden/tree_cases.json (layout and acceptance);
* tree attention: a chain tree is the (separately pinned) VERIFY mask, a star
  tree gives every leaf the attention of a two-token DRAFT block [root, leaf],
  and every node of a random tree equals torch's fp64 attention of its query
  over the context plus its ancestor chain (brute force, tiny sizes);
  relabelling the nodes in another topological order permutes the rows;
* tree acceptance: greedy on a chain tree is the (separately pinned) greedy
  DFlash acceptance; stochastic walks are lossless (the first emitted token
  follows p[root], the second follows p[child] given that child) by chi-square,
  and the root's acceptance rate is the p-mass of its children's tokens.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_cases.json")


def _golden():
    with open(GOLDEN) as fh:
        return json.load(fh)


def test_golden_layout():
    t = _golden()["tree"]
    par = np.array([t["parent"]], np.int32)
    B = par.shape[1]
    table = np.arange(8, dtype=np.int32)[None]
    depth, pos, loc, mask, bad = oracle.tree_prepare(par, [t["seq_len"]], table, 8, 16)
    assert bad == 0
    assert depth[0].tolist() == t["depth"]
    assert pos[0].tolist() == t["positions"]
    assert mask.shape == (1, B, 1) and mask[0, :, 0].tolist() == t["mask"]
    assert loc[0].tolist() == [t["seq_len"] + i for i in range(B)]  # identity paging


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["name"])
def test_golden_accept(case):
    p = np.array(case["p"], np.float32)[None]
    u = None if case.get("greedy") else np.array([case["u"]], np.float32)
    r = oracle.tree_accept([case["block_ids"]], [case["parent"]], p, u, [case["seq_len"]])
    e = case["expected"]
    assert r["accept_len"][0] == e["accept_len"]
    assert r["path"][0].tolist() == e["path"]
    assert r["out_tokens"][0].tolist() == e["out_tokens"]
    assert r["bonus_id"][0] == e["bonus_id"]
    assert r["new_seq_lens"][0] == e["new_seq_len"]


def test_invalid_parent_is_reported_and_made_a_root():
    par = np.array([[5, 0, 3, 1]], np.int32)  # root must be -1; node 2's parent is later
    depth, _, _, mask, bad = oracle.tree_prepare(par, [0], np.zeros((1, 1), np.int32), 1, 8)
    assert bad == 2
    assert depth[0].tolist() == [0, 1, 0, 2] and mask[0, :, 0].tolist() == [1, 3, 4, 11]


# --------------------------------------------------------------- attention
def _attn_inputs(rng, bs, B, Hq, Hkv, D, ps, L):
    L = np.asarray(L, np.int32)
    pages = [(int(l) + B + ps - 1) // ps for l in L]
    total = sum(pages) + 1
    perm = rng.permutation(total).astype(np.int32)
    table = np.full((bs, max(pages)), -1, np.int32)
    at = 0
    for r, n in enumerate(pages):
        table[r, :n] = perm[at:at + n]
        at += n

    def bits(shape):
        x = torch.randn(shape, generator=torch.Generator().manual_seed(int(rng.integers(1 << 30))))
        return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    return (bits((bs * B, Hq, D)), bits((total * ps, Hkv, D)), bits((total * ps, Hkv, D)),
            table, L, total)


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_chain_tree_is_verify_mask():
    rng = np.random.default_rng(1)
    bs, B, Hq, Hkv, D, ps = 2, 6, 4, 2, 16, 4
    q, k, v, table, L, total = _attn_inputs(rng, bs, B, Hq, Hkv, D, ps, [5, 9])
    chain = np.tile(np.arange(-1, B - 1, dtype=np.int32), (bs, 1))
    o_t, l_t = oracle.block_attn_tree(q, k, v, table, L, chain, B, Hq, Hkv, D, ps, 0.25,
                                      num_pages=total)
    o_v, l_v = oracle.block_attn(q, k, v, table, L, B, Hq, Hkv, D, ps, 0.25, 1, num_pages=total)
    np.testing.assert_array_equal(o_t, o_v)
    np.testing.assert_array_equal(l_t, l_v)


def test_star_tree_leaf_is_two_token_draft_block():
    rng = np.random.default_rng(2)
    bs, B, Hq, Hkv, D, ps = 1, 5, 2, 1, 8, 4
    q, k, v, table, L, total = _attn_inputs(rng, bs, B, Hq, Hkv, D, ps, [7])
    star = np.array([[-1, 0, 0, 0, 0]], np.int32)
    o_t, _ = oracle.block_attn_tree(q, k, v, table, L, star, B, Hq, Hkv, D, ps, 0.3,
                                    num_pages=total)
    # leaf i: a cache holding the context, the root and leaf i as a 2-token block
    kf, vf = _f64(k), _f64(v)
    L0 = int(L[0])
    slots = [int(table[0, t // ps]) * ps + t % ps for t in range(L0 + B)]
    for i in range(1, B):
        keep = slots[:L0] + [slots[L0], slots[L0 + i]]
        n2 = len(keep)
        kk = np.zeros(((n2 + ps - 1) // ps * ps, Hkv, D), np.float64)
        vv = np.zeros_like(kk)
        kk[:n2], vv[:n2] = kf[keep], vf[keep]
        to_bits = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16) \
            .view(torch.int16).numpy().view(np.uint16)  # exact: values came from bf16
        qq = np.concatenate([q[0:1], q[i:i + 1]])
        t2 = np.arange(kk.shape[0] // ps, dtype=np.int32)[None]
        o2, _ = oracle.block_attn(qq, to_bits(kk), to_bits(vv), t2, [L0], 2, Hq, Hkv, D, ps, 0.3,
                                  0, num_pages=t2.shape[1])
        np.testing.assert_allclose(o_t[i], o2[1], rtol=1e-12, atol=1e-14)


def _random_tree(rng, B):
    par = np.empty(B, np.int32)
    par[0] = -1
    for i in range(1, B):
        par[i] = rng.integers(0, i)
    return par


def test_random_tree_brute_force_sdpa():
    rng = np.random.default_rng(3)
    bs, B, Hq, Hkv, D, ps = 2, 7, 4, 2, 16, 4
    q, k, v, table, L, total = _attn_inputs(rng, bs, B, Hq, Hkv, D, ps, [6, 11])
    par = np.stack([_random_tree(rng, B) for _ in range(bs)])
    scale = 0.25
    o_t, l_t = oracle.block_attn_tree(q, k, v, table, L, par, B, Hq, Hkv, D, ps, scale,
                                      num_pages=total)
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    G = Hq // Hkv
    for r in range(bs):
        Lr = int(L[r])
        slot = lambda t: int(table[r, t // ps]) * ps + t % ps  # noqa: E731
        for i in range(B):
            chain, n = [], i
            while n >= 0:
                chain.append(n)
                n = int(par[r, n])
            keys = [slot(t) for t in range(Lr)] + [slot(Lr + n) for n in sorted(chain)]
            for j in range(Hq):
                qq = torch.from_numpy(qf[r * B + i, j])[None, None, None]
                kk = torch.from_numpy(kf[keys, j // G])[None, None]
                vv = torch.from_numpy(vf[keys, j // G])[None, None]
                ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale)
                np.testing.assert_allclose(o_t[r * B + i, j], ref[0, 0, 0].numpy(),
                                           rtol=1e-10, atol=1e-12)


def test_relabelling_permutes_rows():
    rng = np.random.default_rng(4)
    bs, B, Hq, Hkv, D, ps = 1, 6, 2, 1, 8, 4
    q, k, v, table, L, total = _attn_inputs(rng, bs, B, Hq, Hkv, D, ps, [5])
    par = np.array([[-1, 0, 0, 1, 2, 1]], np.int32)
    # another topological order of the same tree: new index -> old index
    order = np.array([0, 2, 1, 4, 5, 3])
    inv = np.argsort(order)
    par2 = np.array([[-1] + [int(inv[par[0, order[n]]]) for n in range(1, B)]], np.int32)
    # the block's keys / values and queries follow the nodes
    Lr = int(L[0])
    slots = [int(table[0, t // ps]) * ps + t % ps for t in range(Lr + B)]
    k2, v2 = k.copy(), v.copy()
    for n in range(B):
        k2[slots[Lr + n]] = k[slots[Lr + order[n]]]
        v2[slots[Lr + n]] = v[slots[Lr + order[n]]]
    q2 = q[order]
    o1, _ = oracle.block_attn_tree(q, k, v, table, L, par, B, Hq, Hkv, D, ps, 0.4,
                                   num_pages=total)
    o2, _ = oracle.block_attn_tree(q2, k2, v2, table, L, par2, B, Hq, Hkv, D, ps, 0.4,
                                   num_pages=total)
    np.testing.assert_allclose(o2, o1[order], rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------- acceptance
def _softmax(x):
    e = np.exp(x - x.max(-1, keepdims=True))
    return (e / e.sum(-1, keepdims=True)).astype(np.float32)


def test_greedy_chain_is_dflash_greedy():
    rng = np.random.default_rng(5)
    bs, B, V = 300, 6, 12
    p = _softmax(rng.normal(0, 2, (bs, B, V)))
    ids = rng.integers(0, V, (bs, B)).astype(np.int32)
    # make long accepted prefixes likely: drafts mostly the argmax
    am = p.argmax(-1)
    take = rng.random((bs, B)) < 0.8
    ids[:, 1:] = np.where(take[:, 1:], am[:, :-1], ids[:, 1:])
    chain = np.tile(np.arange(-1, B - 1, dtype=np.int32), (bs, 1))
    seq = rng.integers(0, 100, bs).astype(np.int32)
    t = oracle.tree_accept(ids, chain, p, None, seq)
    d = oracle.spec_accept(ids, p, None, None, None, seq)
    ok = ((t["flags"] & 16) == 0) & ((d["flags"] & 16) == 0)
    np.testing.assert_array_equal(t["accept_len"][ok], d["accept_len"][ok])
    np.testing.assert_array_equal(t["out_tokens"][ok], d["out_tokens"][ok])
    np.testing.assert_array_equal(t["bonus_id"][ok], d["bonus_id"][ok])
    np.testing.assert_array_equal(t["new_seq_lens"][ok], d["new_seq_lens"][ok])
    assert ok.mean() > 0.99


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


@pytest.fixture(scope="module")
def lossless_walks():
    rng = np.random.default_rng(2024)
    n, V = 300_000, 6
    par = np.array([-1, 0, 0, 0, 1, 1, 2, 4], np.int32)
    B = len(par)
    ids = np.array([5, 0, 2, 4, 1, 3, 3, 0], np.int32)
    p = _softmax(rng.normal(0, 1.2, (B, V)))
    u = rng.random((n, B), dtype=np.float32)
    r = oracle.tree_accept(np.tile(ids, (n, 1)), np.tile(par, (n, 1)), p[None], u,
                           np.zeros(n, np.int32), p_strides=(0, V), V=V,
                           nthreads=oracle.max_threads())
    return par, ids, p, r


def test_first_token_follows_root_distribution(lossless_walks):
    par, ids, p, r = lossless_walks
    assert _chi2_ok(np.bincount(r["out_tokens"][:, 0], minlength=p.shape[1]),
                    p[0].astype(np.float64))


def test_second_token_follows_the_accepted_child(lossless_walks):
    par, ids, p, r = lossless_walks
    for child in (1, 2):
        sel = r["path"][:, 1] == child
        assert sel.sum() > 10_000
        assert _chi2_ok(np.bincount(r["out_tokens"][sel, 1], minlength=p.shape[1]),
                        p[child].astype(np.float64))


def test_root_acceptance_rate(lossless_walks):
    par, ids, p, r = lossless_walks
    n = len(r["accept_len"])
    children = [c for c in range(1, len(par)) if par[c] == 0]
    expect = float(p[0, ids[children]].astype(np.float64).sum())
    rate = (r["accept_len"] >= 1).mean()
    assert abs(rate - expect) < 5 * np.sqrt(expect * (1 - expect) / n)
    assert (r["new_seq_lens"] == r["accept_len"] + 1).all()


# ------------------------------------------------- trees above 64 nodes
# The Psi-Spec Tree sampler ((B, K, V) = (16, 32, 32): the top-32 prefixes of
# 15 drafted tokens under the root) gives trees of up to 481 nodes, so the
# ancestor sets span several 64-bit words.
def _mask_words(nodes, W):
    """Words of a node set, written out bit by bit."""
    w = [0] * W
    for n in nodes:
        w[n // 64] |= 1 << (n % 64)
    return w


def test_chain_masks_across_words():
    B = 200
    par = np.arange(-1, B - 1, dtype=np.int32)[None]
    depth, pos, _, mask, bad = oracle.tree_prepare(par, [10], np.zeros((1, 64), np.int32), 1, 8)
    W = 4
    assert mask.shape == (1, B, W)
    for i in (0, 1, 62, 63, 64, 65, 127, 128, 150, 199):
        # closed form: node i's set is {0, ..., i}; full words below i's word
        want = [(2 ** 64 - 1) if 64 * (w + 1) <= i + 1 else
                (0 if 64 * w > i else (1 << (i + 1 - 64 * w)) - 1) for w in range(W)]
        assert [int(x) for x in mask[0, i]] == want, i
    assert depth[0].tolist() == list(range(B)) and pos[0].tolist() == [10 + i for i in range(B)]


def test_star_masks_across_words():
    B = 150
    par = np.zeros((1, B), np.int32)
    par[0, 0] = -1
    _, _, _, mask, _ = oracle.tree_prepare(par, [0], np.zeros((1, 64), np.int32), 1, 8)
    for i in range(1, B):
        assert [int(x) for x in mask[0, i]] == _mask_words([0, i], 3), i


def test_stride_tree_masks_repeat_a_bit_in_every_word():
    # parent(i) = i - 64 for i >= 64, 0 below: node i's ancestors share its bit
    # position in every lower word, so a shifted word index or bit shows
    B = 200
    par = np.array([[-1] + [0 if i < 64 else i - 64 for i in range(1, B)]], np.int32)
    depth, _, _, mask, bad = oracle.tree_prepare(par, [0], np.zeros((1, 64), np.int32), 1, 8)
    assert bad == 0
    for i in (1, 63, 64, 65, 100, 128, 191, 192, 199):
        chain = [0] + [j for j in range(i % 64 or 64, i + 1, 64)]
        assert [int(x) for x in mask[0, i]] == _mask_words(chain, 4), i
        assert depth[0, i] == len(chain) - 1


@pytest.mark.parametrize("shape", ["random", "psi_spec"])
def test_large_tree_masks_follow_the_parent_recurrence(shape):
    from block_diffusion_speculative_attn_gb300 import workloads as wl
    rng = np.random.default_rng(11)
    B = 300
    par = (wl.psi_spec_tree_parents(rng, 2, B) if shape == "psi_spec"
           else np.stack([_random_tree(rng, B) for _ in range(2)]))
    depth, _, _, mask, bad = oracle.tree_prepare(par, [3, 4], np.zeros((2, 64), np.int32), 1, 8)
    assert mask.shape == (2, B, 5)
    for r in range(2):
        for i in range(1, B):
            own = np.array(_mask_words([i], 5), np.uint64)
            np.testing.assert_array_equal(mask[r, i], mask[r, par[r, i]] | own)
            assert sum(bin(int(x)).count("1") for x in mask[r, i]) == depth[r, i] + 1


def test_large_tree_brute_force_sdpa():
    """150 nodes: every node's output is torch's fp64 attention over the
    context and its ancestor chain (the words past the first included)."""
    rng = np.random.default_rng(12)
    bs, B, Hq, Hkv, D, ps = 1, 150, 2, 1, 16, 8
    q, k, v, table, L, total = _attn_inputs(rng, bs, B, Hq, Hkv, D, ps, [37])
    par = _random_tree(rng, B)[None]
    scale = 0.3
    o_t, l_t = oracle.block_attn_tree(q, k, v, table, L, par, B, Hq, Hkv, D, ps, scale,
                                      num_pages=total)
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    Lr = int(L[0])
    slot = lambda t: int(table[0, t // ps]) * ps + t % ps  # noqa: E731
    for i in list(range(0, B, 7)) + [B - 1]:
        chain, n = [], i
        while n >= 0:
            chain.append(n)
            n = int(par[0, n])
        keys = [slot(t) for t in range(Lr)] + [slot(Lr + n) for n in sorted(chain)]
        for j in range(Hq):
            qq = torch.from_numpy(qf[i, j])[None, None, None]
            kk = torch.from_numpy(kf[keys, 0])[None, None]
            vv = torch.from_numpy(vf[keys, 0])[None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale)
            np.testing.assert_allclose(o_t[i, j], ref[0, 0, 0].numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("greedy", [True, False])
def test_long_chain_walk_accepts_every_node(greedy):
    """A 100-node chain whose verifier puts all its mass on the next node's
    token: the walk accepts all 99 nodes below the root and draws the bonus
    from the last node's distribution."""
    B, V = 100, 50
    rng = np.random.default_rng(13)
    ids = rng.integers(0, V, (1, B)).astype(np.int32)
    par = np.arange(-1, B - 1, dtype=np.int32)[None]
    p = np.zeros((1, B, V), np.float32)
    for n in range(B - 1):
        p[0, n, ids[0, n + 1]] = 1.0
    p[0, B - 1, 7] = 1.0
    u = None if greedy else rng.random((1, B)).astype(np.float32)
    r = oracle.tree_accept(ids, par, p, u, [9])
    assert r["accept_len"][0] == B - 1
    assert r["path"][0].tolist() == list(range(B))
    assert r["out_tokens"][0].tolist() == ids[0, 1:].tolist() + [7]
    assert r["bonus_id"][0] == 7 and r["new_seq_lens"][0] == 9 + B
