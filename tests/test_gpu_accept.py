"""GPU parity of bdsa_spec_accept against the fp64 oracle.

Accept lengths, emitted tokens and resampled / bonus tokens must be bit-exact.
The acceptance test is the same IEEE fp32 divide and compare on both sides,
so it must match on every row.  The draw compares u*S with cumulative sums; the
oracle flags rows where u*S lies within 1e-9*S of a boundary of the chosen
token (there two exact-to-1e-13 summation orders may legitimately differ);
those rows are excluded from the comparison and counted, and the count must
stay a tiny fraction of the rows.
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
KEYS = ("accept_len", "commit_len", "bonus_id", "new_seq_lens", "out_tokens")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_cases.json")


def _gpu(acc: wl.AcceptInputs, greedy=False, status=None, sms=0, **kw):
    dev = torch.device("cuda")
    return bdsa.spec_accept(acc.block_ids.to(dev), acc.p.to(dev),
                            None if greedy else acc.q.to(dev), acc.u_acc.to(dev),
                            acc.u_samp.to(dev), acc.seq_lens.to(dev), dev_status=status,
                            sms=sms, **kw)


def _compare(got, want, max_flag_frac=1e-3):
    flags = want["flags"]
    ok = (flags & 2) == 0
    assert (~ok).mean() <= max_flag_frac, f"{(~ok).sum()} flagged rows"
    for k in KEYS:
        g = got[k].cpu().numpy()
        assert (g[ok] == want[k][ok]).all(), (k, np.nonzero((g != want[k]).reshape(len(ok), -1)
                                                           .any(-1) & ok)[0][:10])


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_golden_cases(case):
    dev = torch.device("cuda")
    greedy = bool(case.get("greedy"))
    p = torch.tensor([case["p"]], dtype=torch.float32, device=dev)
    q = None if greedy else torch.tensor([case["q"]], dtype=torch.float32, device=dev)
    out = bdsa.spec_accept(torch.tensor([case["block_ids"]], dtype=torch.int32, device=dev), p, q,
                           torch.tensor([case["u_acc"]], dtype=torch.float32, device=dev),
                           torch.tensor([case["u_samp"]], dtype=torch.float32, device=dev),
                           torch.tensor([case["seq_len"]], dtype=torch.int32, device=dev))
    e = case["expect"]
    assert out["accept_len"].item() == e["accept_len"]
    assert out["commit_len"].item() == e["commit_len"]
    assert out["out_tokens"][0].tolist() == e["out_tokens"]
    assert out["bonus_id"].item() == e["bonus_id"]
    assert out["new_seq_lens"].item() == e["new_seq_len"]


@pytest.mark.parametrize("sms", [0, 1, 4096])
def test_tiny_config(sms):
    cfg = wl.config("tiny")
    acc = wl.make_accept_inputs(cfg, bs=512)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _gpu(acc, status=status, sms=sms)
    want = oracle.spec_accept(acc.block_ids.numpy(), acc.p.numpy(), acc.q.numpy(),
                              acc.u_acc.numpy(), acc.u_samp.numpy(), acc.seq_lens.numpy())
    _compare(got, want)
    assert status.item() == 0


@pytest.mark.parametrize("V", [1, 7, 255, 256, 257, 4099])
@pytest.mark.parametrize("B", [1, 2, 5, 33, 64])
def test_ragged_vocab_and_block(V, B):
    rng = np.random.default_rng(V * 100 + B)
    bs = 64
    p = rng.dirichlet(np.full(V, 0.3), (bs, B)).astype(np.float32)
    q = rng.dirichlet(np.full(V, 0.3), (bs, max(B - 1, 1))).astype(np.float32)[:, :B - 1]
    ids = np.empty((bs, B), np.int32)
    ids[:, 0] = rng.integers(0, V, bs)
    for i in range(1, B):
        c = np.cumsum(q[:, i - 1].astype(np.float64), -1)
        u = rng.random(bs)[:, None] * c[:, -1:]
        ids[:, i] = np.minimum((c <= u).sum(-1), V - 1)
    acc = wl.AcceptInputs(torch.from_numpy(ids), torch.from_numpy(p),
                          torch.from_numpy(np.ascontiguousarray(q)),
                          torch.from_numpy(rng.random((bs, B - 1), dtype=np.float32)),
                          torch.from_numpy(rng.random(bs, dtype=np.float32)),
                          torch.from_numpy(rng.integers(0, 1000, bs).astype(np.int32)))
    for greedy in (False, True):
        got = _gpu(acc, greedy=greedy)
        want = oracle.spec_accept(ids, p, None if greedy else np.ascontiguousarray(q),
                                  acc.u_acc.numpy(), acc.u_samp.numpy(), acc.seq_lens.numpy())
        if greedy:
            ok = (want["flags"] & 16) == 0
            for k in KEYS:
                assert (got[k].cpu().numpy()[ok] == want[k][ok]).all(), k
        else:
            _compare(got, want, max_flag_frac=0.02)


def test_lossless_million_rows_bit_exact():
    """10^6 rows broadcasting one p/q set (stride 0), V = 1000, B = 8: bit-exact with the
    oracle row by row, so the GPU inherits the oracle's chi-square / 1 - TV pins."""
    rng = np.random.default_rng(2024)
    n, B, V = 1_000_000, 8, 1000
    z = 2.0 * rng.standard_normal((B, V))
    p = (np.exp(z - z.max(-1, keepdims=True)))
    p = (p / p.sum(-1, keepdims=True)).astype(np.float32)
    z = 2.0 * rng.standard_normal((B - 1, V))
    q = (np.exp(z - z.max(-1, keepdims=True)))
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    ids = np.empty((n, B), np.int32)
    ids[:, 0] = rng.integers(0, V, n)
    for i in range(1, B):
        c = np.cumsum(q[i - 1].astype(np.float64))
        ids[:, i] = np.minimum(np.searchsorted(c, rng.random(n) * c[-1], side="right"), V - 1)
    u_acc = rng.random((n, B - 1), dtype=np.float32)
    u_samp = rng.random(n, dtype=np.float32)
    sl = np.zeros(n, np.int32)
    dev = torch.device("cuda")
    got = bdsa.spec_accept(torch.from_numpy(ids).to(dev), torch.from_numpy(p).to(dev),
                           torch.from_numpy(q).to(dev), torch.from_numpy(u_acc).to(dev),
                           torch.from_numpy(u_samp).to(dev), torch.from_numpy(sl).to(dev),
                           p_strides=(0, V), q_strides=(0, V), V=V)
    want = oracle.spec_accept(ids, p, q, u_acc, u_samp, sl, p_strides=(0, V), q_strides=(0, V),
                              V=V, nthreads=os.cpu_count() or 1)
    _compare(got, want)


@pytest.mark.parametrize("name", ["qwen3_8b_verify", "uno_1k8k_step", "long_ctx_verify"])
def test_full_size(name):
    cfg = wl.config(name)
    acc = wl.make_accept_inputs(cfg, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = bdsa.spec_accept(acc.block_ids, acc.p, acc.q, acc.u_acc, acc.u_samp, acc.seq_lens,
                           dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    rows = np.arange(cfg.bs) if cfg.bs <= 64 else np.random.default_rng(1).choice(cfg.bs, 48,
                                                                                   replace=False)
    r_t = torch.from_numpy(rows).cuda()
    want = oracle.spec_accept(acc.block_ids[r_t].cpu().numpy(), acc.p[r_t].cpu().numpy(),
                              acc.q[r_t].cpu().numpy(), acc.u_acc[r_t].cpu().numpy(),
                              acc.u_samp[r_t].cpu().numpy(), acc.seq_lens[r_t].cpu().numpy(),
                              nthreads=os.cpu_count() or 1)
    sub = {k: v[r_t] for k, v in got.items()}
    # at these vocabularies no draw falls within 1e-9*S of a boundary: every
    # sampled row is compared
    assert ((want["flags"] & 2) != 0).sum() == 0
    _compare(sub, want, max_flag_frac=0.0)
    c = got["commit_len"].cpu().numpy()
    assert c.min() >= 1 and c.max() <= cfg.B


def test_greedy_full_size():
    cfg = wl.config("qwen3_8b_verify")
    acc = wl.make_accept_inputs(cfg, device="cuda")
    # make roughly half the drafts match the verifier argmax so prefixes vary
    am = acc.p.argmax(-1).to(torch.int32)
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    keep = torch.rand(acc.block_ids[:, 1:].shape, generator=g, device="cuda") < 0.8
    ids = acc.block_ids.clone()
    ids[:, 1:] = torch.where(keep, am[:, :-1], ids[:, 1:])
    got = bdsa.spec_accept(ids, acc.p, None, acc.u_acc, acc.u_samp, acc.seq_lens)
    want = oracle.spec_accept(ids.cpu().numpy(), acc.p.cpu().numpy(), None, acc.u_acc.cpu().numpy(),
                              acc.u_samp.cpu().numpy(), acc.seq_lens.cpu().numpy(),
                              nthreads=os.cpu_count() or 1)
    for k in KEYS:
        assert (got[k].cpu().numpy() == want[k]).all(), k


@pytest.mark.parametrize("V", [1 << 21, (1 << 21) + 1000])
def test_vocab_at_and_beyond_the_cluster_limit(V):
    # 2^21 is the largest vocabulary whose segment totals sit in one CTA's shared
    # memory (64 KB, above the 48 KB default); one more segment takes the path
    # through the global workspace and the last-CTA counter.
    need = bdsa.spec_accept_workspace_bytes(3, 4, V)
    assert (need == 0) == (V <= 1 << 21)
    rng = np.random.default_rng(V)
    bs, B = 3, 4
    p = rng.random((bs, B, V), dtype=np.float32) ** 8
    p /= p.sum(-1, keepdims=True)
    q = p[:, :B - 1] * rng.uniform(0.5, 1.5, (bs, B - 1, V)).astype(np.float32)
    q /= q.sum(-1, keepdims=True)
    ids = np.empty((bs, B), np.int32)
    ids[:, 0] = rng.integers(0, V, bs)
    for i in range(1, B):
        c = np.cumsum(q[:, i - 1].astype(np.float64), -1)
        u = rng.random(bs)[:, None] * c[:, -1:]
        ids[:, i] = np.minimum((c <= u).sum(-1), V - 1)
    acc = wl.AcceptInputs(torch.from_numpy(ids), torch.from_numpy(p), torch.from_numpy(q),
                          torch.from_numpy(rng.random((bs, B - 1), dtype=np.float32)),
                          torch.from_numpy(rng.random(bs, dtype=np.float32)),
                          torch.from_numpy(rng.integers(0, 1000, bs).astype(np.int32)))
    for greedy in (False, True):
        got = _gpu(acc, greedy=greedy)
        want = oracle.spec_accept(ids, p, None if greedy else q, acc.u_acc.numpy(),
                                  acc.u_samp.numpy(), acc.seq_lens.numpy(),
                                  nthreads=os.cpu_count() or 1)
        bad = (want["flags"] & (2 | 16)) != 0
        assert bad.sum() == 0
        for k in KEYS:
            assert (got[k].cpu().numpy() == want[k]).all(), (k, greedy)


def test_bad_draft_id_sets_status():
    cfg = wl.config("tiny")
    acc = wl.make_accept_inputs(cfg, bs=4)
    acc.block_ids[2, 3] = cfg.V + 5
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _gpu(acc, status=status)
    torch.cuda.synchronize()
    assert status.item() == 16
    assert got["accept_len"][2].item() <= 2


@pytest.mark.parametrize("greedy", [False, True])
def test_cuda_graph_capture_and_replay(greedy):
    """The acceptance launch (clusters above the portable 8 CTAs at this shape)
    can be captured in a CUDA graph; replays give the eager call's outputs."""
    cfg = wl.config("qwen3_8b_verify")
    acc = wl.make_accept_inputs(cfg, device="cuda")
    q = None if greedy else acc.q
    want = bdsa.spec_accept(acc.block_ids, acc.p, q, acc.u_acc, acc.u_samp, acc.seq_lens)
    torch.cuda.synchronize()
    out = {k: torch.full_like(v, -7) for k, v in want.items()}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up on the capture stream
        bdsa.spec_accept(acc.block_ids, acc.p, q, acc.u_acc, acc.u_samp, acc.seq_lens, out=out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for v in out.values():
        v.fill_(-7)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bdsa.spec_accept(acc.block_ids, acc.p, q, acc.u_acc, acc.u_samp, acc.seq_lens, out=out)
    for _ in range(2):
        for v in out.values():
            v.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        for k in want:
            assert torch.equal(out[k], want[k]), k
