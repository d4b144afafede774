"""bdsa_spec_accept_noalloc: the acceptance step for callers that cannot give
the library device memory for scratch -- a serving loop whose device memory is
planned once at start-up and may not grow, or a framework that owns the device
allocator and hands the library only the step's own tensors.  It keeps its
scratch in a fixed array inside the library and must give exactly the results
of bdsa_spec_accept (with a workspace) and of the oracle.

Vocabularies above 2^21 are the ones that use that array: the scratch tests
run at V = 2^21 + 1000 and make two calls in a row on different inputs and
batch sizes, so that the second call starts from the first call's leftovers.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes
import os

import numpy as np
import pytest
import torch

import block_diffusion_speculative_attn_gb300 as bdsa
import oracle
from block_diffusion_speculative_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
KEYS = ("accept_len", "commit_len", "out_tokens", "bonus_id", "new_seq_lens")
SCRATCH_BYTES = 8 << 20  # the fixed array's size, as declared in include/bdsa.h
V_SCRATCH = (1 << 21) + 1000  # just past the vocabularies that need no scratch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(acc: wl.AcceptInputs, greedy: bool):
    """Call the entry point through the C ABI; outputs are pre-filled with -7
    so that anything left unwritten shows."""
    L = bdsa.lib()
    bs, B = acc.block_ids.shape
    V = acc.p.shape[-1]
    out = {k: torch.full((bs,), -7, dtype=torch.int32, device="cuda")
           for k in ("accept_len", "commit_len", "bonus_id", "new_seq_lens")}
    out["out_tokens"] = torch.full((bs, B), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = None if greedy else acc.q
    st = L.bdsa_spec_accept_noalloc(
        _ptr(acc.block_ids), _ptr(acc.p), B * V, V, _ptr(q), (B - 1) * V if q is not None else 0,
        V if q is not None else 0, _ptr(acc.u_acc), _ptr(acc.u_samp), _ptr(acc.seq_lens), bs, B, V,
        _ptr(out["accept_len"]), _ptr(out["commit_len"]), _ptr(out["out_tokens"]),
        _ptr(out["bonus_id"]), _ptr(out["new_seq_lens"]), 0, _ptr(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out, status


def _with_workspace(acc: wl.AcceptInputs, greedy: bool):
    bs, B = acc.block_ids.shape
    ws_bytes = bdsa.spec_accept_workspace_bytes(bs, B, acc.p.shape[-1])
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    return bdsa.spec_accept(acc.block_ids, acc.p, None if greedy else acc.q, acc.u_acc,
                            acc.u_samp, acc.seq_lens, workspace=ws)


def _wide_vocab_inputs(bs: int, B: int, V: int, seed: int) -> wl.AcceptInputs:
    """Peaked p (u^8, normalised), q = p with +-50% noise, drafts drawn from q."""
    rng = np.random.default_rng(seed)
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
    return wl.AcceptInputs(torch.from_numpy(ids), torch.from_numpy(p), torch.from_numpy(q),
                           torch.from_numpy(rng.random((bs, B - 1), dtype=np.float32)),
                           torch.from_numpy(rng.random(bs, dtype=np.float32)),
                           torch.from_numpy(rng.integers(0, 1000, bs).astype(np.int32)))


def _to(acc: wl.AcceptInputs, dev) -> wl.AcceptInputs:
    return wl.AcceptInputs(*(t.to(dev) for t in (acc.block_ids, acc.p, acc.q, acc.u_acc,
                                                   acc.u_samp, acc.seq_lens)))


@pytest.mark.parametrize("greedy", [False, True])
def test_fixed_scratch_two_calls_in_a_row(greedy):
    """Two calls in a row through the fixed array (bs 3, then bs 4 on other
    inputs): each equals the workspace entry point and the oracle bit for bit."""
    B = 4
    for bs, seed in ((3, 101), (4, 202)):
        need = bdsa.spec_accept_workspace_bytes(bs, B, V_SCRATCH)
        assert 0 < need <= SCRATCH_BYTES  # this problem does go through the array
        host = _wide_vocab_inputs(bs, B, V_SCRATCH, seed)
        acc = _to(host, "cuda")
        st, got, status = _noalloc(acc, greedy)
        assert st == 0, bdsa.STATUS.get(st, st)
        want = _with_workspace(acc, greedy)
        torch.cuda.synchronize()
        assert status.item() == 0
        for k in KEYS:
            assert torch.equal(got[k], want[k]), (k, bs)
        ref = oracle.spec_accept(host.block_ids.numpy(), host.p.numpy(),
                                 None if greedy else host.q.numpy(), host.u_acc.numpy(),
                                 host.u_samp.numpy(), host.seq_lens.numpy(),
                                 nthreads=os.cpu_count() or 1)
        # no draw within the summation-order band of a boundary (flag bit 2);
        # greedy ties (bit 16) are settled by the lowest index on both sides
        assert ((ref["flags"] & 2) == 0).all()
        for k in KEYS:
            assert (got[k].cpu().numpy() == ref[k]).all(), (k, bs)


@pytest.mark.parametrize("greedy", [False, True])
def test_no_scratch_needed_two_calls_in_a_row(greedy):
    """At the Qwen3-8B vocabulary (151936 <= 2^21) nothing uses the array; two
    calls in a row still equal the workspace entry point."""
    cfg = wl.config("qwen3_8b_verify")
    for seed in (11, 12):
        acc = wl.make_accept_inputs(cfg, device="cuda", seed=seed)
        st, got, status = _noalloc(acc, greedy)
        assert st == 0, bdsa.STATUS.get(st, st)
        want = bdsa.spec_accept(acc.block_ids, acc.p, None if greedy else acc.q, acc.u_acc,
                                acc.u_samp, acc.seq_lens)
        torch.cuda.synchronize()
        assert status.item() == 0
        for k in KEYS:
            assert torch.equal(got[k], want[k]), k


def test_small_vocab_and_batch_reuse():
    cfg = wl.config("tiny")
    for bs in (3, 300):
        acc = wl.make_accept_inputs(cfg, device="cuda", bs=bs)
        st, got, _ = _noalloc(acc, False)
        assert st == 0
        want = bdsa.spec_accept(acc.block_ids, acc.p, acc.q, acc.u_acc, acc.u_samp,
                                acc.seq_lens)
        torch.cuda.synchronize()
        for k in KEYS:
            assert torch.equal(got[k], want[k]), k


def _raw(bs, B, V, ptr):
    L = bdsa.lib()
    return L.bdsa_spec_accept_noalloc(ptr, ptr, 0, 0, ptr, 0, 0, ptr, ptr, ptr, bs, B, V, ptr,
                                      ptr, ptr, ptr, ptr, 0, None, None)


def test_rejects_problems_larger_than_the_fixed_scratch():
    # 128 rows of 2^22 need ~17 MB of scratch; the array holds 8 MiB
    bs, B, V = 128, 16, 1 << 22
    assert bdsa.lib().bdsa_spec_accept_workspace_bytes(bs, B, V, 0) > SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    assert _raw(bs, B, V, _ptr(dummy)) == 4  # BDSA_WORKSPACE_TOO_SMALL, nothing launched


def test_argument_errors_match_the_workspace_entry_point():
    # the argument checks come before the size check: B > 64 is UNSUPPORTED and
    # a null pointer INVALID_ARG, even for a problem too large for the array
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    assert _raw(128, 65, 1 << 22, _ptr(dummy)) == 2
    assert _raw(128, 16, 1 << 22, None) == 1
    assert _raw(-1, 4, 1000, _ptr(dummy)) == 1
    assert _raw(0, 4, 1000, _ptr(dummy)) == 0
