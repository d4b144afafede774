"""GPU parity of bdsa_block_attn_paged_append (the block's own K/V written into
the paged cache in the same launch as the block attention that reads them).

Before each call the block's cache slots hold NaN, so a kernel that read a
stale row instead of the one it wrote would fail.  The caches after the call
must equal the oracle's append bit for bit (nothing else written), and the
output must match the fp64 oracle's attention on the appended caches within
the attention tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from block_diffusion_speculative_attn_gb300 import workloads as wl
from gpu_helpers import DevAttn, assert_attn_close, oracle_attn_requests

pytestmark = pytest.mark.gpu
DRAFT, VERIFY = wl.DRAFT, wl.VERIFY
FORCE_SPLIT = 4096


def _cfg(name, bs, Hq, Hkv, D, B, ps, seq_lens, seed=91):
    return wl.StepConfig(name, bs, Hq, Hkv, D, B, ps, tuple(seq_lens), (DRAFT, VERIFY), seed=seed)


SHAPES = [
    # name, Hq, Hkv, D, B, page_size, seq_lens
    ("tiny_like", 2, 1, 64, 8, 16, (200, 256)),
    ("ragged_d128_g2", 4, 2, 128, 8, 16, (0, 1, 127, 120, 129, 300)),
    ("qwen_like_g4_b16", 32, 8, 128, 16, 64, (1000, 37)),
    ("llada_like_rows128", 16, 4, 128, 32, 32, (513, 700)),
    ("decode_b1_d64", 8, 8, 64, 1, 8, (50, 400, 0)),
    ("b64_big_pages", 2, 1, 64, 64, 256, (333,)),
    ("block_straddles_tiles", 4, 2, 128, 16, 8, (120, 250)),
]


def _block_rows(inp, cfg):
    _, _, cache_loc, bad = oracle.prepare_block(np.zeros(cfg.bs, np.int32), inp.seq_lens,
                                                inp.block_table, inp.num_pages, cfg.B,
                                                cfg.page_size, 0)
    return cache_loc.reshape(-1), bad


def _new_kv(cfg, seed):
    g = torch.Generator().manual_seed(seed)
    shape = (cfg.bs * cfg.B, cfg.Hkv, cfg.D)
    return (torch.randn(shape, generator=g).to(torch.bfloat16),
            torch.randn(shape, generator=g).to(torch.bfloat16))


def _run_append(inp, cfg, k_cache, v_cache, k_new, v_new, mode, sms=0, status=None):
    import block_diffusion_speculative_attn_gb300 as bdsa
    dev = torch.device("cuda")
    kc, vc = k_cache.to(dev), v_cache.to(dev)
    lse = torch.full((inp.q.shape[0], cfg.Hq), float("nan"), dtype=torch.float32, device=dev)
    out = bdsa.block_attn_paged(inp.q.to(dev), kc, vc, torch.from_numpy(inp.block_table).to(dev),
                                torch.from_numpy(inp.seq_lens).to(dev), B=cfg.B,
                                page_size=cfg.page_size, scale=inp.scale, mode=mode,
                                max_ctx_len=inp.max_ctx_len, num_pages=inp.num_pages, lse=lse,
                                dev_status=status, sms=sms, k_new=k_new.to(dev),
                                v_new=v_new.to(dev))
    torch.cuda.synchronize()
    return out, lse, kc.cpu(), vc.cpu()


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("mode", [DRAFT, VERIFY])
@pytest.mark.parametrize("sms", [0, 5, FORCE_SPLIT])
def test_append_then_attend(shape, mode, sms):
    name, Hq, Hkv, D, B, ps, lens = shape
    cfg = _cfg(name, len(lens), Hq, Hkv, D, B, ps, lens)
    inp = wl.make_attn_inputs(cfg, extra_pages=2)
    loc, bad = _block_rows(inp, cfg)
    assert bad == 0
    k_cache, v_cache = inp.k_cache.clone(), inp.v_cache.clone()
    k_cache[torch.from_numpy(loc)] = float("nan")
    v_cache[torch.from_numpy(loc)] = float("nan")
    k_new, v_new = _new_kv(cfg, 7 + mode)
    k_exp, v_exp = oracle.append_block_kv(wl.bf16_bits(k_cache), wl.bf16_bits(v_cache),
                                          wl.bf16_bits(k_new), wl.bf16_bits(v_new),
                                          inp.block_table, inp.seq_lens, B, ps, inp.num_pages)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, kc, vc = _run_append(inp, cfg, k_cache, v_cache, k_new, v_new, mode, sms, status)
    assert status.item() == 0
    np.testing.assert_array_equal(wl.bf16_bits(kc), k_exp)
    np.testing.assert_array_equal(wl.bf16_bits(vc), v_exp)
    ref, ref_lse = oracle.block_attn(wl.bf16_bits(inp.q), k_exp, v_exp, inp.block_table,
                                     inp.seq_lens, B, Hq, Hkv, D, ps, inp.scale, mode,
                                     num_pages=inp.num_pages, nthreads=8)
    assert_attn_close(out, ref, lse, ref_lse, tag=f"append {name} mode={mode} sms={sms}")


def test_append_skips_pages_outside_the_pool():
    cfg = _cfg("badpage", 3, 8, 2, 128, 8, 16, (100, 200, 50))
    inp = wl.make_attn_inputs(cfg)
    table = inp.block_table.copy()
    table[1, 200 // 16] = inp.num_pages + 7  # request 1's block page is outside the pool
    bad_inp = wl.AttnInputs(cfg, inp.seq_lens, table, inp.num_pages, inp.q, inp.k_cache,
                            inp.v_cache, inp.scale)
    k_new, v_new = _new_kv(cfg, 3)
    k_exp, v_exp = oracle.append_block_kv(wl.bf16_bits(inp.k_cache), wl.bf16_bits(inp.v_cache),
                                          wl.bf16_bits(k_new), wl.bf16_bits(v_new), table,
                                          inp.seq_lens, cfg.B, cfg.page_size, inp.num_pages)
    for sms in (0, 5, FORCE_SPLIT):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, lse, kc, vc = _run_append(bad_inp, cfg, inp.k_cache, inp.v_cache, k_new, v_new,
                                       VERIFY, sms, status)
        assert status.item() == 16
        np.testing.assert_array_equal(wl.bf16_bits(kc), k_exp)
        np.testing.assert_array_equal(wl.bf16_bits(vc), v_exp)
        o = out.float().cpu().numpy()
        assert (o[cfg.B:2 * cfg.B] == 0).all()
        assert (lse[cfg.B:2 * cfg.B] == float("-inf")).all()


def test_append_full_size_verify():
    """Qwen3-8B-shaped verify batch in the benchmark's launch configuration: the
    whole caches compared bit for bit, outputs of sampled requests against the
    oracle."""
    cfg = wl.config("qwen3_8b_verify")
    inp = wl.make_attn_inputs(cfg)
    loc, bad = _block_rows(inp, cfg)
    assert bad == 0
    k_cache, v_cache = inp.k_cache.clone(), inp.v_cache.clone()
    k_cache[torch.from_numpy(loc)] = float("nan")
    v_cache[torch.from_numpy(loc)] = float("nan")
    k_new, v_new = _new_kv(cfg, 11)
    k_exp, v_exp = oracle.append_block_kv(wl.bf16_bits(k_cache), wl.bf16_bits(v_cache),
                                          wl.bf16_bits(k_new), wl.bf16_bits(v_new),
                                          inp.block_table, inp.seq_lens, cfg.B, cfg.page_size,
                                          inp.num_pages)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, kc, vc = _run_append(inp, cfg, k_cache, v_cache, k_new, v_new, VERIFY, 0, status)
    assert status.item() == 0
    np.testing.assert_array_equal(wl.bf16_bits(kc), k_exp)
    np.testing.assert_array_equal(wl.bf16_bits(vc), v_exp)
    d = DevAttn.__new__(DevAttn)
    d.inp, d.q = inp, inp.q.cuda()
    d.k, d.v = kc.cuda(), vc.cuda()
    rng = np.random.default_rng(4)
    reqs = sorted({0, cfg.bs - 1, int(rng.integers(cfg.bs))})
    ref, ref_lse, rows = oracle_attn_requests(d, reqs, VERIFY)
    assert_attn_close(out[torch.from_numpy(rows).cuda()], ref, lse[torch.from_numpy(rows).cuda()],
                      ref_lse, tag="append qwen3_8b_verify")
