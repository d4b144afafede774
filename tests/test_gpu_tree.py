"""GPU parity of tree verify ("Unlocking Lossless Speedups in LLMs via Discrete
Diffusion", Psi-Spec Tree sampler; "SGLang dLLM / LLaDA 2.0", "Attention
Mask"): bdsa_tree_prepare (bit-exact), bdsa_block_attn_paged_tree (the
attention tolerance against the fp64 oracle; a chain tree against the VERIFY
oracle and the VERIFY call) and bdsa_tree_accept (bit-exact, rows whose draw the oracle flags
as within 1e-9 of a boundary excluded and counted).
"""
import dataclasses
import json
import os

import numpy as np
import pytest
import torch

import block_diffusion_speculative_attn_gb300 as bdsa
import oracle
from block_diffusion_speculative_attn_gb300 import workloads as wl
from gpu_helpers import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_cases.json")
KEYS = bdsa.TREE_KEYS + ("path", "out_tokens")


def _t(x, dtype):
    return torch.as_tensor(np.ascontiguousarray(x), dtype=dtype, device=DEV)


# ------------------------------------------------------------------ prepare
@pytest.mark.parametrize("B", [1, 2, 7, 32, 64, 65, 200, 481, 512])
def test_prepare_matches_oracle(B):
    rng = np.random.default_rng(B)
    bs, ps = 97, 16
    par = wl.random_tree_parents(rng, bs, B)
    par[3, B - 1] = B + 5 if B > 1 else 4   # invalid parents: reported, made roots
    par[5, 0] = 0
    seq = rng.integers(0, 3000, bs).astype(np.int32)
    table, num_pages = wl.paging_for(seq, B, ps, rng, extra_pages=2)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = bdsa.tree_prepare(_t(par, torch.int32), _t(seq, torch.int32), _t(table, torch.int32),
                            num_pages, ps, dev_status=status)
    want = oracle.tree_prepare(par, seq, table, num_pages, ps)
    for g, w in zip(got[:3], want[:3]):
        np.testing.assert_array_equal(g.cpu().numpy(), w)
    np.testing.assert_array_equal(got[3].cpu().numpy().view(np.uint64), want[3])
    assert want[4] > 0 and status.item() == 16


# ---------------------------------------------------------------- attention
def _tree_attn_case(cfg, n_nodes, seed, chain=False, shape="bushy", device="cpu"):
    c = dataclasses.replace(cfg, B=n_nodes)
    inp = wl.make_attn_inputs(c, device=device, seed=seed)
    rng = np.random.default_rng(seed)
    if chain:
        par = np.tile(np.arange(-1, n_nodes - 1, dtype=np.int32), (c.bs, 1))
    elif shape == "psi_spec":
        par = wl.psi_spec_tree_parents(rng, c.bs, n_nodes)
    else:
        par = wl.random_tree_parents(rng, c.bs, n_nodes)
    return c, inp, par


def _run_tree_attn(c, inp, par, sms=0):
    q, k, v = inp.q.to(DEV), inp.k_cache.to(DEV), inp.v_cache.to(DEV)
    bt = torch.from_numpy(inp.block_table).to(DEV)
    sl = torch.from_numpy(inp.seq_lens).to(DEV)
    _, _, _, mask = bdsa.tree_prepare(_t(par, torch.int32), sl, bt, inp.num_pages, c.page_size)
    lse = torch.empty((q.shape[0], c.Hq), dtype=torch.float32, device=DEV)
    out = bdsa.block_attn_paged(q, k, v, bt, sl, B=c.B, page_size=c.page_size, scale=inp.scale,
                                mode=bdsa.VERIFY, max_ctx_len=inp.max_ctx_len,
                                num_pages=inp.num_pages, lse=lse, tree_mask=mask, sms=sms)
    torch.cuda.synchronize()
    return out, lse, (q, k, v, bt, sl)


def _oracle_tree(c, inp, par):
    return oracle.block_attn_tree(wl.bf16_bits(inp.q), wl.bf16_bits(inp.k_cache),
                                  wl.bf16_bits(inp.v_cache), inp.block_table, inp.seq_lens, par,
                                  c.B, c.Hq, c.Hkv, c.D, c.page_size, inp.scale,
                                  num_pages=inp.num_pages, nthreads=oracle.max_threads())


@pytest.mark.parametrize("n_nodes", [1, 5, 16, 32, 33, 100, 481])
def test_tree_attention_matches_oracle(n_nodes):
    """G = 4: one tile of 4 * nodes rows up to 32 nodes, then row tiles of 32
    nodes (two at 33 nodes, sixteen at 481, the last holding one node)."""
    cfg = dataclasses.replace(wl.config("tiny"), bs=3, Hq=8, Hkv=2, D=128, page_size=16,
                              ctx=((0, 300),))
    c, inp, par = _tree_attn_case(cfg, n_nodes, 11 + n_nodes)
    out, lse, _ = _run_tree_attn(c, inp, par)
    ref, ref_lse = _oracle_tree(c, inp, par)
    assert_attn_close(out, ref, lse, ref_lse, tag=f"tree {n_nodes}")


@pytest.mark.parametrize("sms", [0, 7])
@pytest.mark.parametrize("D,Hq,Hkv,n_nodes", [(64, 2, 2, 200), (128, 16, 2, 100),
                                              (128, 6, 2, 150), (128, 8, 2, 512),
                                              (64, 256, 2, 3)])
def test_row_tiles_match_oracle(D, Hq, Hkv, n_nodes, sms):
    """Trees of more than 128 / G nodes in row tiles of floor(128 / G) nodes:
    G = 1 (two tiles of 128 nodes), G = 8 (seven of 16), G = 3 (four of 42,
    126-row tiles), G = 4 at the largest tree (sixteen of 32), G = 128 (one
    node a tile); contexts up to 1500 keys, and with sms = 7 every row tile
    cut between CTAs (merged partials)."""
    cfg = dataclasses.replace(wl.config("tiny"), bs=3, Hq=Hq, Hkv=Hkv, D=D, page_size=32,
                              ctx=((0, 1500),))
    c, inp, par = _tree_attn_case(cfg, n_nodes, 3 * n_nodes + Hq)
    out, lse, _ = _run_tree_attn(c, inp, par, sms=sms)
    ref, ref_lse = _oracle_tree(c, inp, par)
    assert_attn_close(out, ref, lse, ref_lse, tag=f"row tiles G={Hq // Hkv} nodes={n_nodes}")


def test_long_chain_tree_is_the_verify_mask():
    """A 200-node chain (seven row tiles of 32 nodes at G = 4) masks exactly as
    VERIFY with B = 200: it matches the fp64 VERIFY oracle."""
    cfg = dataclasses.replace(wl.config("tiny"), bs=2, Hq=8, Hkv=2, D=128, page_size=16,
                              ctx=((100, 900),))
    c, inp, par = _tree_attn_case(cfg, 200, 21, chain=True)
    out, lse, _ = _run_tree_attn(c, inp, par)
    ref, ref_lse = oracle.block_attn(wl.bf16_bits(inp.q), wl.bf16_bits(inp.k_cache),
                                     wl.bf16_bits(inp.v_cache), inp.block_table, inp.seq_lens,
                                     c.B, c.Hq, c.Hkv, c.D, c.page_size, inp.scale, bdsa.VERIFY,
                                     num_pages=inp.num_pages, nthreads=oracle.max_threads())
    assert_attn_close(out, ref, lse, ref_lse, tag="200-node chain vs verify oracle")


@pytest.mark.parametrize("D,G", [(64, 1), (128, 4), (128, 8)])
def test_chain_tree_is_the_verify_mask(D, G):
    """A chain tree masks exactly as VERIFY: the tree call matches the fp64
    VERIFY oracle, and the GPU VERIFY call, within the attention tolerance."""
    cfg = dataclasses.replace(wl.config("tiny"), bs=5, Hq=2 * G, Hkv=2, D=D, page_size=16,
                              ctx=((0, 700),))
    c, inp, par = _tree_attn_case(cfg, 16, 7, chain=True)
    out_t, lse_t, (q, k, v, bt, sl) = _run_tree_attn(c, inp, par)
    ref, ref_lse = oracle.block_attn(wl.bf16_bits(inp.q), wl.bf16_bits(inp.k_cache),
                                     wl.bf16_bits(inp.v_cache), inp.block_table, inp.seq_lens,
                                     c.B, c.Hq, c.Hkv, c.D, c.page_size, inp.scale, bdsa.VERIFY,
                                     num_pages=inp.num_pages, nthreads=8)
    assert_attn_close(out_t, ref, lse_t, ref_lse, tag="chain tree vs verify oracle")
    lse_v = torch.empty_like(lse_t)
    out_v = bdsa.block_attn_paged(q, k, v, bt, sl, B=c.B, page_size=c.page_size,
                                  scale=inp.scale, mode=bdsa.VERIFY, max_ctx_len=inp.max_ctx_len,
                                  num_pages=inp.num_pages, lse=lse_v)
    torch.cuda.synchronize()
    assert_attn_close(out_t, out_v.float().cpu().numpy().reshape(ref.shape), lse_t,
                      lse_v.cpu().numpy().reshape(ref_lse.shape), tag="chain tree vs verify")


@pytest.mark.parametrize("n_nodes,shape", [(32, "bushy"), (481, "psi_spec"), (256, "psi_spec")])
def test_qwen3_8b_shaped_tree_attention(n_nodes, shape):
    """Batch 32, 32/8 heads, contexts U[1024, 4096]: 32-node trees (G * nodes =
    128: one M = 128 tile), and trees shaped like the Psi-Spec Tree sampler's
    (B, K, V) = (16, 32, 32) -- 32 prefixes of 15 tokens under the root, 481
    nodes (sixteen row tiles), or 256; the oracle checks four requests."""
    cfg = wl.config("qwen3_8b_verify")
    c, inp, par = _tree_attn_case(cfg, n_nodes, 5, shape=shape)
    out, lse, (q, k, v, bt, sl) = _run_tree_attn(c, inp, par)
    reqs = [0, 10, 21, 31]
    # compact copy of the sampled requests' pages for the oracle
    ps = c.page_size
    need = [(int(inp.seq_lens[r]) + c.B + ps - 1) // ps for r in reqs]
    pages = np.concatenate([inp.block_table[r, :n] for r, n in zip(reqs, need)])
    kc = inp.k_cache.view(-1, ps, c.Hkv, c.D)[torch.from_numpy(pages.astype(np.int64))]
    vc = inp.v_cache.view(-1, ps, c.Hkv, c.D)[torch.from_numpy(pages.astype(np.int64))]
    table = np.full((len(reqs), max(need)), -1, np.int32)
    at = 0
    for j, n in enumerate(need):
        table[j, :n] = np.arange(at, at + n)
        at += n
    rows = torch.cat([torch.arange(r * c.B, (r + 1) * c.B) for r in reqs])
    ref, ref_lse = oracle.block_attn_tree(
        wl.bf16_bits(inp.q[rows]), wl.bf16_bits(kc.reshape(-1, c.Hkv, c.D)),
        wl.bf16_bits(vc.reshape(-1, c.Hkv, c.D)), table, inp.seq_lens[reqs], par[reqs], c.B,
        c.Hq, c.Hkv, c.D, ps, inp.scale, num_pages=at, nthreads=oracle.max_threads())
    assert_attn_close(out[rows.to(DEV)], ref, lse[rows.to(DEV)], ref_lse, tag="qwen tree")


# --------------------------------------------------------------- acceptance
def _compare(got, want, max_flag_frac=1e-3):
    ok = (want["flags"] & 18) == 0
    assert (~ok).mean() <= max_flag_frac, f"{(~ok).sum()} flagged rows"
    for k in KEYS:
        g = got[k].cpu().numpy()
        bad = (g != want[k]).reshape(len(ok), -1).any(-1) & ok
        assert not bad.any(), (k, np.nonzero(bad)[0][:10])
    return int((~ok).sum())


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_golden_accept(case):
    p = _t(np.array(case["p"], np.float32)[None], torch.float32)
    u = None if case.get("greedy") else _t([case["u"]], torch.float32)
    r = bdsa.tree_accept(_t([case["block_ids"]], torch.int32), _t([case["parent"]], torch.int32),
                         p, u, _t([case["seq_len"]], torch.int32))
    e = case["expected"]
    assert r["accept_len"].item() == e["accept_len"]
    assert r["path"][0].tolist() == e["path"]
    assert r["out_tokens"][0].tolist() == e["out_tokens"]
    assert r["bonus_id"].item() == e["bonus_id"]
    assert r["new_seq_lens"].item() == e["new_seq_len"]


@pytest.mark.parametrize("greedy", [False, True])
@pytest.mark.parametrize("V", [1, 7, 257, 4099])
@pytest.mark.parametrize("n_nodes", [1, 2, 9, 64, 65, 300])
def test_random_trees(n_nodes, V, greedy):
    cfg = dataclasses.replace(wl.config("tiny"), V=V)
    x = wl.make_tree_inputs(cfg, n_nodes, bs=64, seed=n_nodes * 31 + V)
    u = None if greedy else x.u
    got = bdsa.tree_accept(x.block_ids.to(DEV), _t(x.parent, torch.int32), x.p.to(DEV),
                           None if u is None else u.to(DEV), x.seq_lens.to(DEV))
    want = oracle.tree_accept(x.block_ids.numpy(), x.parent, x.p.numpy(),
                              None if u is None else u.numpy(), x.seq_lens.numpy())
    _compare(got, want, max_flag_frac=0.05)


@pytest.mark.parametrize("sms", [0, 1, 4096])
def test_chunking_does_not_change_results(sms):
    cfg = dataclasses.replace(wl.config("tiny"), V=30000)
    x = wl.make_tree_inputs(cfg, 16, bs=24, seed=3)
    got = bdsa.tree_accept(x.block_ids.to(DEV), _t(x.parent, torch.int32), x.p.to(DEV),
                           x.u.to(DEV), x.seq_lens.to(DEV), sms=sms)
    want = oracle.tree_accept(x.block_ids.numpy(), x.parent, x.p.numpy(), x.u.numpy(),
                              x.seq_lens.numpy())
    _compare(got, want, max_flag_frac=0.05)


def test_invalid_parent_is_reported_and_never_a_child():
    cfg = dataclasses.replace(wl.config("tiny"), V=50)
    x = wl.make_tree_inputs(cfg, 6, bs=4, seed=9)
    par = x.parent.copy()
    par[1, 3] = 9
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = bdsa.tree_accept(x.block_ids.to(DEV), _t(par, torch.int32), x.p.to(DEV),
                           x.u.to(DEV), x.seq_lens.to(DEV), dev_status=status)
    want = oracle.tree_accept(x.block_ids.numpy(), par, x.p.numpy(), x.u.numpy(),
                              x.seq_lens.numpy())
    _compare(got, want, max_flag_frac=0.5)
    assert status.item() == 16


def test_qwen3_8b_shaped_tree_acceptance():
    """Batch 32, 32-node trees, vocabulary 151936, drafter close to the
    verifier: every row against the oracle."""
    cfg = wl.config("qwen3_8b_verify")
    x = wl.make_tree_inputs(cfg, 32, device=DEV)
    got = bdsa.tree_accept(x.block_ids, _t(x.parent, torch.int32), x.p, x.u, x.seq_lens)
    torch.cuda.synchronize()
    want = oracle.tree_accept(x.block_ids.cpu().numpy(), x.parent, x.p.cpu().numpy(),
                              x.u.cpu().numpy(), x.seq_lens.cpu().numpy(),
                              nthreads=oracle.max_threads())
    _compare(got, want, max_flag_frac=2 / 32)
    assert got["accept_len"].float().mean().item() >= 1.0


@pytest.mark.parametrize("greedy", [False, True])
def test_psi_spec_sized_tree_acceptance(greedy):
    """Eight requests with 481-node trees shaped like the Psi-Spec Tree
    sampler's (B, K, V) = (16, 32, 32) at vocabulary 151936: every row against
    the oracle (the walk is at most 16 nodes deep)."""
    cfg = wl.config("qwen3_8b_verify")
    x = wl.make_tree_inputs(cfg, 481, device=DEV, bs=8, shape="psi_spec")
    u = None if greedy else x.u
    got = bdsa.tree_accept(x.block_ids, _t(x.parent, torch.int32), x.p, u, x.seq_lens)
    torch.cuda.synchronize()
    want = oracle.tree_accept(x.block_ids.cpu().numpy(), x.parent, x.p.cpu().numpy(),
                              None if u is None else u.cpu().numpy(), x.seq_lens.cpu().numpy(),
                              nthreads=oracle.max_threads())
    _compare(got, want, max_flag_frac=1 / 8)
    assert got["accept_len"].max().item() <= 15
