"""Pins for the oracle's block attention (CPU only).

The oracle (oracle/bdsa_oracle.c) follows the mask definition of "SGLang dLLM /
LLaDA 2.0", section "Attention Mask": every block query sees the whole cached
context; inside the block the mask is a rectangle in block-diffusion (DRAFT)
mode and a token-causal trapezoid in chunked-prefill (VERIFY) mode, which is
also the causal verify of "From DFlash to dLLM Self-Spec (IV)", section 4.4.1.
These tests tie it to things other than itself:

* torch's scaled_dot_product_attention on CPU in fp64: VERIFY equals the last B
  rows of token-causal prefill over the concatenated context+block sequence,
  DRAFT equals unmasked attention of the B queries over all keys, and B = 1 is
  ordinary decode attention;
* closed forms: constant V rows give o = v; Q = 0 gives the mean of the allowed
  V rows and lse = log(number of allowed keys);
* invariance to how pages are permuted in the pool and block table.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_speculative_attn_gb300 import workloads as wl

DRAFT, VERIFY = 0, 1


def _bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 and return their uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _instance(seq_lens, B, Hq, Hkv, D, ps, seed, perm_seed=None, extra_pages=3):
    """Contiguous per-request sequences, then scattered into a shuffled page pool."""
    rng = np.random.default_rng(seed)
    bs = len(seq_lens)
    seqs_k, seqs_v, qs = [], [], []
    for L in seq_lens:
        n = L + B
        seqs_k.append(_bf16(rng.standard_normal((n, Hkv, D))))
        seqs_v.append(_bf16(rng.standard_normal((n, Hkv, D))))
        qs.append(_bf16(rng.standard_normal((n, Hq, D))))  # queries for every position
    prng = np.random.default_rng(seed + 1 if perm_seed is None else perm_seed)
    table, num_pages = wl.paging_for(np.asarray(seq_lens, np.int32), B, ps, prng, extra_pages)
    slots = num_pages * ps
    # fill unused slots with NaN bit patterns: the oracle must never read them
    kc = np.full((slots, Hkv, D), 0x7FC0, np.uint16)
    vc = np.full((slots, Hkv, D), 0x7FC0, np.uint16)
    for r, L in enumerate(seq_lens):
        for t in range(L + B):
            slot = table[r, t // ps] * ps + t % ps
            kc[slot] = seqs_k[r][t]
            vc[slot] = seqs_v[r][t]
    qb = np.concatenate([qs[r][L:L + B] for r, L in enumerate(seq_lens)], axis=0)
    return dict(seqs_k=seqs_k, seqs_v=seqs_v, qs=qs, table=table, num_pages=num_pages,
                kc=kc, vc=vc, qb=qb, seq_lens=np.asarray(seq_lens, np.int32))


def _sdpa(q, k, v, G, scale, causal):
    """torch CPU SDPA in fp64.  q [Tq, Hq, D], k/v [Tk, Hkv, D] -> [Tq, Hq, D]."""
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal,
                                                         scale=scale)
    return o[0].permute(1, 0, 2).numpy()


CASES = [
    # seq_lens, B, Hq, Hkv, D, page_size
    ((9, 14), 4, 4, 2, 16, 4),
    ((0, 5, 33), 3, 6, 3, 8, 8),
    ((17,), 8, 2, 1, 32, 16),
    ((40, 3), 5, 8, 2, 16, 2),
]


@pytest.mark.parametrize("case", CASES)
def test_verify_is_causal_prefill_tail(case):
    seq_lens, B, Hq, Hkv, D, ps = case
    inst = _instance(seq_lens, B, Hq, Hkv, D, ps, seed=11)
    scale = 1.0 / math.sqrt(D)
    out, _ = oracle.block_attn(inst["qb"], inst["kc"], inst["vc"], inst["table"],
                               inst["seq_lens"], B, Hq, Hkv, D, ps, scale, VERIFY,
                               num_pages=inst["num_pages"])
    for r, L in enumerate(seq_lens):
        ref = _sdpa(_bits_to_f64(inst["qs"][r]), _bits_to_f64(inst["seqs_k"][r]),
                    _bits_to_f64(inst["seqs_v"][r]), Hq // Hkv, scale, causal=True)[L:L + B]
        np.testing.assert_allclose(out[r * B:(r + 1) * B], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", CASES)
def test_draft_is_unmasked_attention(case):
    seq_lens, B, Hq, Hkv, D, ps = case
    inst = _instance(seq_lens, B, Hq, Hkv, D, ps, seed=12)
    scale = 0.37
    out, _ = oracle.block_attn(inst["qb"], inst["kc"], inst["vc"], inst["table"],
                               inst["seq_lens"], B, Hq, Hkv, D, ps, scale, DRAFT,
                               num_pages=inst["num_pages"])
    for r, L in enumerate(seq_lens):
        ref = _sdpa(_bits_to_f64(inst["qs"][r][L:L + B]), _bits_to_f64(inst["seqs_k"][r]),
                    _bits_to_f64(inst["seqs_v"][r]), Hq // Hkv, scale, causal=False)
        np.testing.assert_allclose(out[r * B:(r + 1) * B], ref, rtol=0, atol=1e-12)


def test_block_size_one_is_decode():
    seq_lens, B, Hq, Hkv, D, ps = (31, 0, 64), 1, 4, 2, 16, 8
    inst = _instance(seq_lens, B, Hq, Hkv, D, ps, seed=13)
    scale = 1.0 / math.sqrt(D)
    outs = [oracle.block_attn(inst["qb"], inst["kc"], inst["vc"], inst["table"],
                              inst["seq_lens"], B, Hq, Hkv, D, ps, scale, m,
                              num_pages=inst["num_pages"])[0] for m in (DRAFT, VERIFY)]
    np.testing.assert_array_equal(outs[0], outs[1])
    for r, L in enumerate(seq_lens):
        ref = _sdpa(_bits_to_f64(inst["qs"][r][L:L + 1]), _bits_to_f64(inst["seqs_k"][r]),
                    _bits_to_f64(inst["seqs_v"][r]), Hq // Hkv, scale, causal=False)
        np.testing.assert_allclose(outs[0][r:r + 1], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("mode", [DRAFT, VERIFY])
def test_zero_query_closed_form(mode):
    """Q = 0: every allowed key has score 0, so o = mean of allowed V and lse = log n."""
    seq_lens, B, Hq, Hkv, D, ps = (5, 0, 23), 6, 4, 1, 8, 4
    inst = _instance(seq_lens, B, Hq, Hkv, D, ps, seed=14)
    qb = np.zeros_like(inst["qb"])
    out, lse = oracle.block_attn(qb, inst["kc"], inst["vc"], inst["table"], inst["seq_lens"],
                                 B, Hq, Hkv, D, ps, 0.5, mode, num_pages=inst["num_pages"])
    G = Hq // Hkv
    for r, L in enumerate(seq_lens):
        v = _bits_to_f64(inst["seqs_v"][r])
        for i in range(B):
            n = L + B if mode == DRAFT else L + i + 1
            for j in range(Hq):
                np.testing.assert_allclose(out[r * B + i, j], v[:n, j // G].mean(0), atol=1e-13)
                assert abs(lse[r * B + i, j] - math.log(n)) < 1e-13


def test_constant_values_closed_form():
    seq_lens, B, Hq, Hkv, D, ps = (12, 7), 4, 2, 2, 8, 4
    inst = _instance(seq_lens, B, Hq, Hkv, D, ps, seed=15)
    vconst = _bf16(np.linspace(-2, 2, D))
    vc = inst["vc"].copy()
    vc[:] = vconst[None, None, :]
    for mode in (DRAFT, VERIFY):
        out, _ = oracle.block_attn(inst["qb"], inst["kc"], vc, inst["table"], inst["seq_lens"],
                                   B, Hq, Hkv, D, ps, 0.3, mode, num_pages=inst["num_pages"])
        np.testing.assert_allclose(out, np.broadcast_to(_bits_to_f64(vconst), out.shape),
                                   atol=1e-13)


def test_page_permutation_invariance():
    seq_lens, B, Hq, Hkv, D, ps = (21, 40), 5, 4, 2, 16, 4
    a = _instance(seq_lens, B, Hq, Hkv, D, ps, seed=16, perm_seed=100)
    b = _instance(seq_lens, B, Hq, Hkv, D, ps, seed=16, perm_seed=200)
    assert not np.array_equal(a["table"], b["table"])
    for mode in (DRAFT, VERIFY):
        oa, la = oracle.block_attn(a["qb"], a["kc"], a["vc"], a["table"], a["seq_lens"], B, Hq,
                                   Hkv, D, ps, 0.25, mode, num_pages=a["num_pages"])
        ob, lb = oracle.block_attn(b["qb"], b["kc"], b["vc"], b["table"], b["seq_lens"], B, Hq,
                                   Hkv, D, ps, 0.25, mode, num_pages=b["num_pages"])
        np.testing.assert_array_equal(oa, ob)
        np.testing.assert_array_equal(la, lb)


def test_mode_row_relations():
    """Last block row sees the same keys in both modes; VERIFY row 0 is decode over L+1 keys."""
    seq_lens, B, Hq, Hkv, D, ps = (19, 2), 6, 4, 2, 16, 4
    inst = _instance(seq_lens, B, Hq, Hkv, D, ps, seed=17)
    args = (inst["qb"], inst["kc"], inst["vc"], inst["table"], inst["seq_lens"], B, Hq, Hkv, D,
            ps, 0.25)
    od, _ = oracle.block_attn(*args, DRAFT, num_pages=inst["num_pages"])
    ov, _ = oracle.block_attn(*args, VERIFY, num_pages=inst["num_pages"])
    for r, L in enumerate(seq_lens):
        np.testing.assert_array_equal(od[r * B + B - 1], ov[r * B + B - 1])
        ref = _sdpa(_bits_to_f64(inst["qs"][r][L:L + 1]), _bits_to_f64(inst["seqs_k"][r][:L + 1]),
                    _bits_to_f64(inst["seqs_v"][r][:L + 1]), Hq // Hkv, 0.25, causal=False)
        np.testing.assert_allclose(ov[r * B:r * B + 1], ref, atol=1e-12)


def test_out_of_range_page_is_reported():
    seq_lens, B, Hq, Hkv, D, ps = (8,), 4, 2, 1, 8, 4
    inst = _instance(seq_lens, B, Hq, Hkv, D, ps, seed=18)
    table = inst["table"].copy()
    table[0, 1] = inst["num_pages"] + 5
    with pytest.raises(ValueError):
        oracle.block_attn(inst["qb"], inst["kc"], inst["vc"], table, inst["seq_lens"], B, Hq,
                          Hkv, D, ps, 0.3, VERIFY, num_pages=inst["num_pages"])
