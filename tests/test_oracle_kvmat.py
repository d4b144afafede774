"""Pins of the oracle's KV materialisation of the committed rows ("From DFlash
to dLLM Self-Spec (II)", section 2.2.6, and the DFlash engineering notes:
projection across draft layers, K RMS norm, RoPE, write at the verify slots)
against things other than itself:

* hand-worked cases under tests/golden/kv_materialize_cases.json (rotation
  pairing and sign, gain, eps, the [layer][K, V][head] weight layout);
* V against numpy's fp64 matmul of the widened bf16 operands;
* closed forms of the K path: with an identity table (cos 1, sin 0) and unit
  gains every K head vector has mean square ms / (ms + eps) ~ 1, and scaling x
  leaves K unchanged while V scales with it; the table rotation keeps every
  (d, d + D/2) pair's length; with the RoPE table, the dot product of two
  rotated copies of one row depends only on the position difference;
* only committed rows are written; a bad slot or position is skipped and
  counted.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_speculative_attn_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_materialize_cases.json")


def _bits(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_golden_cases(case):
    k, v, st = oracle.kv_materialize(
        _bits(case["hidden"]), case["commit_len"], case["positions"], case["cache_loc"],
        _bits(case["w_kv"]), _bits(case["k_norm_w"]), np.array(case["cos"], np.float32),
        np.array(case["sin"], np.float32), case["eps"], case["B"], case["n_layers"],
        case["Hkv"], case["D"], case["num_slots"])
    e = case["expected"]
    assert st.tolist() == e["status"]
    rows = [i for i, s in enumerate(e["status"]) if s == 1]
    np.testing.assert_allclose(k[rows], np.array(e["k"]), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(v[rows], np.array(e["v"]), rtol=1e-6, atol=1e-7)
    assert np.isnan(k[[i for i in range(len(st)) if st[i] != 1]]).all()


def _small(seed, bs=3, B=4, H=48, n_layers=2, Hkv=2, D=8, max_pos=64):
    rng = np.random.default_rng(seed)
    hidden = _bits(rng.standard_normal((bs * B, H)))
    w = _bits(rng.standard_normal((n_layers, 2, Hkv * D, H)) / np.sqrt(H))
    g = _bits(1 + 0.1 * rng.standard_normal((n_layers, D)))
    commit = rng.integers(1, B + 1, bs).astype(np.int32)
    pos = rng.integers(0, max_pos, bs * B).astype(np.int32)
    loc = rng.permutation(64)[: bs * B].astype(np.int32)
    return rng, hidden, w, g, commit, pos, loc


def test_v_is_the_matmul_and_only_committed_rows_are_written():
    rng, hidden, w, g, commit, pos, loc = _small(1)
    bs, B, H, L, Hkv, D = 3, 4, 48, 2, 2, 8
    cos, sin = wl.rope_tables(64, D)
    k, v, st = oracle.kv_materialize(hidden, commit, pos, loc, w, g, cos.numpy(), sin.numpy(),
                                     1e-6, B, L, Hkv, D, 64)
    want = np.einsum("lvoc,rc->rlvo", _f64(w).reshape(L, 2, Hkv * D, H), _f64(hidden))
    committed = (np.arange(bs * B) % B) < np.repeat(commit, B)
    assert (st == committed.astype(np.int32)).all()
    np.testing.assert_allclose(v[committed].reshape(-1, L, Hkv * D),
                               want[committed][:, :, 1], rtol=1e-12, atol=1e-12)
    assert np.isnan(v[~committed]).all() and np.isnan(k[~committed]).all()


def test_norm_closed_form_and_scale_invariance():
    rng, hidden, w, g, commit, pos, loc = _small(2)
    B, L, Hkv, D, eps = 4, 2, 2, 8, 1e-6
    ones = _bits(np.ones((L, D)))
    ident_c = np.ones((64, D // 2), np.float32)
    ident_s = np.zeros((64, D // 2), np.float32)
    k, v, st = oracle.kv_materialize(hidden, commit, pos, loc, w, ones, ident_c, ident_s, eps,
                                     B, L, Hkv, D, 64)
    ok = st == 1
    # mean square after the norm: ms / (ms + eps), with ms the projection's
    ms_after = (k[ok] ** 2).mean(-1)
    k_raw = np.einsum("lhdc,rc->rlhd", _f64(w)[:, 0].reshape(L, Hkv, D, -1), _f64(hidden)[ok])
    ms = (k_raw ** 2).mean(-1)
    np.testing.assert_allclose(ms_after, ms / (ms + eps), rtol=1e-12)
    # x -> 2x (exact in bf16): K unchanged up to eps, V doubled
    k2, v2, _ = oracle.kv_materialize(_bits(2 * _f64(hidden)), commit, pos, loc, w, ones,
                                      ident_c, ident_s, 0.0, B, L, Hkv, D, 64)
    k0, v0, _ = oracle.kv_materialize(hidden, commit, pos, loc, w, ones, ident_c, ident_s, 0.0,
                                      B, L, Hkv, D, 64)
    np.testing.assert_allclose(k2[ok], k0[ok], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(v2[ok], 2 * v0[ok], rtol=1e-12)


def test_rotation_keeps_pair_lengths_and_gain_applies_before_it():
    rng, hidden, w, g, commit, pos, loc = _small(3)
    B, L, Hkv, D = 4, 2, 2, 8
    cos, sin = wl.rope_tables(64, D)
    ident_c = np.ones((64, D // 2), np.float32)
    ident_s = np.zeros((64, D // 2), np.float32)
    kr, _, st = oracle.kv_materialize(hidden, commit, pos, loc, w, g, cos.numpy(), sin.numpy(),
                                      1e-6, B, L, Hkv, D, 64)
    kn, _, _ = oracle.kv_materialize(hidden, commit, pos, loc, w, g, ident_c, ident_s, 1e-6, B,
                                     L, Hkv, D, 64)
    ok = st == 1
    h = D // 2
    c2 = cos.numpy().astype(np.float64) ** 2 + sin.numpy().astype(np.float64) ** 2
    scale = c2[pos[ok]][:, None, None, :]  # |table row| is 1 up to fp32 rounding
    lr = kr[ok][..., :h] ** 2 + kr[ok][..., h:] ** 2
    ln = kn[ok][..., :h] ** 2 + kn[ok][..., h:] ** 2
    np.testing.assert_allclose(lr, ln * scale, rtol=1e-12, atol=1e-15)
    # rows at position 0 are not rotated
    z = ok & (pos == 0)
    if z.any():
        np.testing.assert_allclose(kr[z], kn[z], rtol=0, atol=0)


def test_relative_position_property():
    """One row at positions m, n and m + t, n + t: <K(m), K(n)> = <K(m+t), K(n+t)>."""
    rng, hidden, w, g, _, _, _ = _small(4, bs=1, B=4)
    B, L, Hkv, D = 4, 2, 2, 8
    hidden = np.repeat(hidden[:1], 4, axis=0)
    cos, sin = wl.rope_tables(256, D, base=100.0)
    pos = np.array([3, 11, 103, 111], np.int32)  # (3, 11) and (103, 111): same gap
    k, _, st = oracle.kv_materialize(hidden, [4], pos, np.arange(4, dtype=np.int32), w, g,
                                     cos.numpy(), sin.numpy(), 1e-6, B, L, Hkv, D, 4)
    assert (st == 1).all()
    a = (k[0] * k[1]).sum(-1)
    b = (k[2] * k[3]).sum(-1)
    np.testing.assert_allclose(a, b, rtol=1e-5, atol=1e-6)
    # and it does change with the gap
    c = (k[0] * k[3]).sum(-1)
    assert np.abs(c - a).max() > 1e-3


def test_bad_slot_or_position_is_skipped_and_counted():
    rng, hidden, w, g, commit, pos, loc = _small(5)
    B, L, Hkv, D = 4, 2, 2, 8
    commit = np.array([4, 4, 4], np.int32)
    loc = loc.copy()
    pos = pos.copy()
    loc[1] = -1
    loc[5] = 64          # == num_slots
    pos[9] = 64          # == max_pos
    cos, sin = wl.rope_tables(64, D)
    k, v, st = oracle.kv_materialize(hidden, commit, pos, loc, w, g, cos.numpy(), sin.numpy(),
                                     1e-6, B, L, Hkv, D, 64)
    assert st.tolist().count(-1) == 3 and st[1] == st[5] == st[9] == -1
    assert np.isnan(k[[1, 5, 9]]).all()
    assert np.isfinite(k[st == 1]).all()


def test_commit_len_is_clamped():
    rng, hidden, w, g, _, pos, loc = _small(6)
    B, L, Hkv, D = 4, 2, 2, 8
    cos, sin = wl.rope_tables(64, D)
    _, _, st = oracle.kv_materialize(hidden, [-3, 9, 2], pos, loc, w, g, cos.numpy(),
                                     sin.numpy(), 1e-6, B, L, Hkv, D, 64)
    assert st.reshape(3, B).tolist() == [[0, 0, 0, 0], [1, 1, 1, 1], [1, 1, 0, 0]]
