"""Shared plumbing for the GPU parity tests: move seeded inputs to the device,
gather a few requests into a compact cache for the oracle, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from block_diffusion_speculative_attn_gb300 import workloads as wl

# Tolerance against the fp64 oracle for bf16 inputs with fp32 accumulation.
ATTN_MAX_ABS = 1e-2
ATTN_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


class DevAttn:
    """An AttnInputs instance with its tensors on the GPU."""

    def __init__(self, inp: wl.AttnInputs, dev="cuda"):
        self.inp = inp
        self.q = inp.q.to(dev)
        self.k = inp.k_cache.to(dev)
        self.v = inp.v_cache.to(dev)
        self.bt = torch.from_numpy(inp.block_table).to(dev)
        self.sl = torch.from_numpy(inp.seq_lens).to(dev)


def run_attn(d: DevAttn, mode: int, sms: int = 0, status=None, lse=True):
    import block_diffusion_speculative_attn_gb300 as bdsa
    cfg = d.inp.cfg
    lse_t = None
    if lse:
        lse_t = torch.full((d.q.shape[0], cfg.Hq), float("nan"), dtype=torch.float32,
                           device=d.q.device)
    out = bdsa.block_attn_paged(d.q, d.k, d.v, d.bt, d.sl, B=cfg.B, page_size=cfg.page_size,
                                scale=d.inp.scale, mode=mode, max_ctx_len=d.inp.max_ctx_len,
                                num_pages=d.inp.num_pages, lse=lse_t, dev_status=status, sms=sms)
    torch.cuda.synchronize()
    return out, lse_t


def oracle_attn_full(inp: wl.AttnInputs, mode: int, nthreads: int = 8):
    cfg = inp.cfg
    return oracle.block_attn(wl.bf16_bits(inp.q), wl.bf16_bits(inp.k_cache),
                             wl.bf16_bits(inp.v_cache), inp.block_table, inp.seq_lens, cfg.B,
                             cfg.Hq, cfg.Hkv, cfg.D, cfg.page_size, inp.scale, mode,
                             num_pages=inp.num_pages, nthreads=nthreads)


def oracle_attn_requests(d: DevAttn, reqs, mode: int, nthreads: int = 16):
    """Oracle output for a subset of requests, from a compact copy of their pages."""
    inp, cfg = d.inp, d.inp.cfg
    ps = cfg.page_size
    reqs = list(reqs)
    need = [(int(inp.seq_lens[r]) + cfg.B + ps - 1) // ps for r in reqs]
    pages = np.concatenate([inp.block_table[r, :n] for r, n in zip(reqs, need)]).astype(np.int64)
    idx = torch.from_numpy(pages).to(d.k.device)
    kc = d.k.view(-1, ps, cfg.Hkv, cfg.D)[idx].reshape(-1, cfg.Hkv, cfg.D)
    vc = d.v.view(-1, ps, cfg.Hkv, cfg.D)[idx].reshape(-1, cfg.Hkv, cfg.D)
    table = np.full((len(reqs), max(need)), -1, np.int32)
    at = 0
    for j, n in enumerate(need):
        table[j, :n] = np.arange(at, at + n, dtype=np.int32)
        at += n
    rows = torch.cat([torch.arange(r * cfg.B, (r + 1) * cfg.B) for r in reqs]).to(d.q.device)
    q = d.q[rows]
    out, lse = oracle.block_attn(wl.bf16_bits(q), wl.bf16_bits(kc), wl.bf16_bits(vc), table,
                                 inp.seq_lens[reqs], cfg.B, cfg.Hq, cfg.Hkv, cfg.D, ps, inp.scale,
                                 mode, num_pages=at, nthreads=nthreads)
    return out, lse, rows.cpu().numpy()


def assert_attn_close(got: torch.Tensor, ref: np.ndarray, lse_got=None, lse_ref=None, tag=""):
    g = got.float().cpu().numpy().reshape(ref.shape)
    assert np.isfinite(g).all(), f"{tag}: non-finite output"
    err = np.abs(g - ref)
    assert err.max() <= ATTN_MAX_ABS, f"{tag}: max abs err {err.max():.3e}"
    assert err.mean() <= ATTN_MEAN_ABS, f"{tag}: mean abs err {err.mean():.3e}"
    if lse_got is not None and lse_ref is not None:
        lg = lse_got.cpu().numpy().reshape(lse_ref.shape)
        le = np.abs(lg - lse_ref)
        assert le.max() <= LSE_MAX_ABS, f"{tag}: lse max abs err {le.max():.3e}"
    return float(err.max()), float(err.mean())
