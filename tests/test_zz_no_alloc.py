"""bdsa_spec_accept_noalloc: the acceptance step for callers that cannot give
the library device memory for scratch (a memory plan fixed at start-up, a CUDA
graph capture in progress, a framework that owns the allocator).  It uses a
fixed scratch array inside the library and must give exactly the results of
bdsa_spec_accept.  This file is collected last on purpose: if it fails, a run
that stops at the first failure has already run every other test."""
import ctypes

import pytest
import torch

import block_diffusion_speculative_attn_gb300 as bdsa
from block_diffusion_speculative_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
KEYS = ("accept_len", "commit_len", "out_tokens", "bonus_id", "new_seq_lens")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(acc: wl.AcceptInputs, greedy: bool):
    """Call the entry point through the C ABI with outputs allocated here."""
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


@pytest.mark.parametrize("greedy", [False, True])
def test_matches_workspace_entry_point_on_two_calls(greedy):
    cfg = wl.config("qwen3_8b_verify")
    for seed in (11, 12):  # two calls in a row, different inputs
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


def test_rejects_problems_larger_than_the_fixed_scratch():
    L = bdsa.lib()
    # vocabularies above 2^21 keep their segment totals in global scratch:
    # 128 rows of 2^22 needs ~17 MB, the array holds 8 MiB
    bs, B, V = 128, 16, 1 << 22
    assert L.bdsa_spec_accept_workspace_bytes(bs, B, V, 0) > (8 << 20)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    st = L.bdsa_spec_accept_noalloc(_ptr(dummy), _ptr(dummy), 0, 0, _ptr(dummy), 0, 0,
                                    _ptr(dummy), _ptr(dummy), _ptr(dummy), bs, B, V, _ptr(dummy),
                                    _ptr(dummy), _ptr(dummy), _ptr(dummy), _ptr(dummy), 0, None,
                                    None)
    assert st == 4  # BDSA_WORKSPACE_TOO_SMALL, nothing launched
