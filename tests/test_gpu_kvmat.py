"""GPU parity of bdsa_kv_materialize (the draft K/V of the committed rows:
"From DFlash to dLLM Self-Spec (II)", section 2.2.6 and the DFlash
engineering notes) against the fp64 oracle.

Outputs are bf16 rounded once from an fp32 result (fp32 accumulation of bf16
products on the tensor cores, fp32 norm and rotation), so every written
element must lie within one bf16 ulp of the fp64 value, plus 2^-14 of its head
vector's RMS for the accumulation error next to values near zero.  Slots that must not be written are filled with a
NaN pattern first and must keep it bit for bit.
"""
import numpy as np
import pytest
import torch

import block_diffusion_speculative_attn_gb300 as bdsa
import oracle
from block_diffusion_speculative_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENTINEL = 0x7FC1  # a quiet-NaN bf16 pattern the kernel never writes


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ulp_err(got_bits, ref):
    """|got - ref| in units of the allowed error: one bf16 ulp of |ref| (2^-8
    relative) plus 2^-14 of the head vector's RMS, the room the fp32
    accumulation of up to a few thousand products needs next to values near
    zero."""
    got = _f64(got_bits)
    rms = np.sqrt((ref ** 2).mean(-1, keepdims=True))
    return np.abs(got - ref) / (np.abs(ref) * 2.0 ** -8 + rms * 2.0 ** -14)


class Case:
    def __init__(self, x: wl.KvMatInputs):
        self.x = x

    def layout(self, page_size):
        """positions L_r + i and slots page * ps + (L_r + i) % ps, from the
        separately pinned oracle prepare_block."""
        x = self.x
        bs = x.commit_len.shape[0]
        _, pos, loc, bad = oracle.prepare_block(np.zeros(bs, np.int32), x.seq_lens,
                                                x.block_table, x.num_pages, x.B, page_size, 0)
        assert bad == 0
        self.positions, self.cache_loc = pos.reshape(-1), loc.reshape(-1)
        self.num_slots = x.num_pages * page_size
        return self

    def compact(self, seed):
        """positions L_r + i, slots a permutation of the bs*B block rows (a
        pool holding just this block's rows)."""
        x = self.x
        bs = x.commit_len.shape[0]
        self.positions = (x.seq_lens[:, None] + np.arange(x.B)[None, :]).astype(np.int32)
        self.positions = self.positions.reshape(-1)
        self.cache_loc = np.random.default_rng(seed).permutation(bs * x.B).astype(np.int32)
        self.num_slots = bs * x.B
        return self


def _run(case: Case, commit=None, positions=None, cache_loc=None, status=None):
    x = case.x
    L, Hkv, D = x.n_layers, x.Hkv, x.D
    commit = x.commit_len if commit is None else torch.as_tensor(commit, dtype=torch.int32)
    pos = case.positions if positions is None else positions
    loc = case.cache_loc if cache_loc is None else cache_loc
    kc = torch.full((L, case.num_slots, Hkv, D), SENTINEL, dtype=torch.int16,
                    device=DEV).view(torch.bfloat16)
    vc = kc.clone()
    bdsa.kv_materialize(x.hidden.to(DEV), commit.to(DEV),
                        torch.from_numpy(np.ascontiguousarray(pos)).to(DEV),
                        torch.from_numpy(np.ascontiguousarray(loc)).to(DEV), x.w_kv.to(DEV),
                        x.k_norm_w.to(DEV), x.rope_cos.to(DEV), x.rope_sin.to(DEV), kc, vc,
                        B=x.B, eps=x.eps, dev_status=status)
    torch.cuda.synchronize()
    return _bits(kc), _bits(vc), commit.cpu().numpy(), pos, loc


def _check(case, got, rows=None, nthreads=None):
    x = case.x
    kb, vb, commit, pos, loc = got
    hidden_bits = _bits(x.hidden)
    k_ref, v_ref, st = oracle.kv_materialize(
        hidden_bits, commit, pos, loc, _bits(x.w_kv), _bits(x.k_norm_w), x.rope_cos.numpy(),
        x.rope_sin.numpy(), x.eps, x.B, x.n_layers, x.Hkv, x.D, case.num_slots,
        nthreads=nthreads or oracle.max_threads())
    written = np.zeros(case.num_slots, bool)
    written[loc[st == 1]] = True
    worst = 0.0
    for row in np.nonzero(st == 1)[0]:
        if rows is not None and row not in rows:
            continue
        s = loc[row]
        ek = _ulp_err(kb[:, s], k_ref[row])
        ev = _ulp_err(vb[:, s], v_ref[row])
        worst = max(worst, float(ek.max()), float(ev.max()))
    assert worst <= 1.0, f"max error {worst:.3f} bf16 ulp"
    # nothing else was written
    assert (kb[:, ~written] == SENTINEL).all() and (vb[:, ~written] == SENTINEL).all()
    return st, worst


def _small(bs=3, B=4, H=256, n_layers=2, Hkv=2, seed=0, commit=None, max_ctx=300):
    cfg = wl.StepConfig("kvmat_small", bs, Hkv * 2, Hkv, 128, B, 16, ((0, max_ctx),), (1,))
    x = wl.make_kvmat_inputs(cfg, n_layers=n_layers, H=H, seed=seed, bs=bs, max_ctx=max_ctx)
    if commit is not None:
        x.commit_len = torch.as_tensor(np.asarray(commit, np.int32))
    return Case(x).layout(16)


@pytest.mark.parametrize("H", [128, 256, 1024])
def test_small_matches_oracle(H):
    case = _small(H=H, seed=H)
    st, worst = _check(case, _run(case))
    assert (st == 1).sum() == int(case.x.commit_len.sum())


@pytest.mark.parametrize("commit", [[0, 0, 0], [4, 4, 4], [1, 0, 3]])
def test_commit_lengths(commit):
    case = _small(seed=7, commit=commit)
    st, _ = _check(case, _run(case))
    assert (st == 1).sum() == sum(commit)


def test_several_passes_over_the_weights():
    """More than 128 committed rows: three passes (128, 128, 64 rows)."""
    case = _small(bs=40, B=8, H=256, n_layers=1, Hkv=2, seed=3, commit=[8] * 40)
    st, _ = _check(case, _run(case))
    assert (st == 1).sum() == 320


@pytest.mark.parametrize("n_rows", [1, 15, 16, 17, 31, 33, 63, 64, 65, 127, 128, 129])
def test_ragged_row_counts(n_rows):
    B = 16
    bs = (n_rows + B - 1) // B
    commit = [B] * (n_rows // B) + ([n_rows % B] if n_rows % B else [])
    case = _small(bs=bs, B=B, H=128, n_layers=1, Hkv=1, seed=n_rows, commit=commit)
    st, _ = _check(case, _run(case))
    assert (st == 1).sum() == n_rows


def test_bad_slot_or_position_is_skipped_and_reported():
    case = _small(seed=11, commit=[4, 4, 4])
    loc = case.cache_loc.copy()
    pos = case.positions.copy()
    loc[1] = -1
    loc[6] = case.num_slots
    pos[9] = case.x.rope_cos.shape[0]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _run(case, positions=pos, cache_loc=loc, status=status)
    st, _ = _check(case, got)
    assert status.item() == 16 and (st == -1).sum() == 3


def test_qwen3_8b_shaped_drafter():
    """Batch 32, B = 16, hidden 4096, five draft layers of 8 KV heads x 128:
    the launch the benchmark times; the oracle checks four requests' rows."""
    cfg = wl.config("qwen3_8b_verify")
    x = wl.make_kvmat_inputs(cfg, n_layers=5, H=4096)
    case = Case(x).compact(5)
    got = _run(case)
    # the oracle computes only the sampled requests' rows (others uncommitted)
    commit = got[2].copy()
    keep = np.zeros_like(commit)
    keep[[0, 9, 20, 31]] = commit[[0, 9, 20, 31]]
    kb, vb, _, pos, loc = got
    k_ref, v_ref, st = oracle.kv_materialize(
        _bits(x.hidden), keep, pos, loc, _bits(x.w_kv), _bits(x.k_norm_w), x.rope_cos.numpy(),
        x.rope_sin.numpy(), x.eps, x.B, x.n_layers, x.Hkv, x.D, case.num_slots,
        nthreads=oracle.max_threads())
    worst, where = 0.0, None
    for row in np.nonzero(st == 1)[0]:
        s = loc[row]
        for name, got, ref in (("k", kb[:, s], k_ref[row]), ("v", vb[:, s], v_ref[row])):
            e = _ulp_err(got, ref)
            if e.max() > worst:
                i = np.unravel_index(int(e.argmax()), e.shape)
                worst, where = float(e.max()), (name, row, i, float(_f64(got)[i]), ref[i])
    assert worst <= 1.0, f"max error {worst:.3f} of the tolerance at {where}"
    # every committed row of every request was written, nothing else
    written = np.zeros(case.num_slots, bool)
    for r in range(cfg.bs):
        written[loc[r * cfg.B: r * cfg.B + commit[r]]] = True
    assert (kb[:, written] != SENTINEL).all() and (vb[:, written] != SENTINEL).all()
    assert (kb[:, ~written] == SENTINEL).all() and (vb[:, ~written] == SENTINEL).all()
