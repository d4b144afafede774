"""GPU parity of bdsa_block_attn_paged against the fp64 oracle.

Tolerance (bf16 inputs, fp32 accumulation, bf16 output): max-abs 1e-2 and
mean-abs 1e-3 on the output, 1e-3 on the natural-log lse.  Cases span several
128-key tiles with ragged tails, L = 0, every supported G*B packing, page sizes
below, at and above the 128-key tile, both masks, and both the single-split and
the split-KV (combine) paths.  Full-size workloads are checked on sampled
requests.
"""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_attn_gb300 import workloads as wl
from gpu_helpers import (DevAttn, assert_attn_close, oracle_attn_full, oracle_attn_requests,
                         run_attn)

pytestmark = pytest.mark.gpu
DRAFT, VERIFY = wl.DRAFT, wl.VERIFY
FORCE_SPLIT = 4096  # an SM count that makes the planner split every unit's KV range
# A grid of 5 CTAs: units are cut into several pieces, and (being no larger than
# the device) the 64-row tile merges them in the attention launch, in the CTA
# holding each cut unit's first tile; FORCE_SPLIT (more CTAs than SMs) keeps
# the separate merge launch.
OWNER = 5
SMS = [0, OWNER, FORCE_SPLIT]


def _cfg(name, bs, Hq, Hkv, D, B, ps, seq_lens, seed=77):
    return wl.StepConfig(name, bs, Hq, Hkv, D, B, ps, tuple(seq_lens), (DRAFT, VERIFY), seed=seed)


SHAPES = [
    # name, Hq, Hkv, D, B, page_size, seq_lens
    ("ragged_d128_g2", 4, 2, 128, 8, 16, (0, 1, 127, 120, 129, 300)),
    ("qwen_like_g4_b16", 32, 8, 128, 16, 64, (1000, 37)),
    ("llada_like_rows128", 16, 4, 128, 32, 32, (513, 700)),
    ("long_like_g8", 64, 8, 128, 16, 64, (259, 1500)),
    ("decode_b1_d64", 8, 8, 64, 1, 8, (50, 400, 0)),
    ("b64_big_pages", 2, 1, 64, 64, 256, (333,)),
    ("odd_g3_b3", 6, 2, 64, 3, 128, (240, 17)),
    # 63 tiles in one unit: with the forced split it is cut into more pieces than
    # the merge kernel lists up front
    ("long_unit_many_pieces", 2, 1, 64, 4, 64, (8000,)),
]


@pytest.fixture(scope="module")
def dev():
    import block_diffusion_speculative_attn_gb300 as bdsa
    bdsa.lib()
    return torch.device("cuda")


@pytest.mark.parametrize("mode", [DRAFT, VERIFY])
@pytest.mark.parametrize("sms", SMS)
def test_tiny_config(dev, mode, sms):
    inp = wl.make_attn_inputs(wl.config("tiny"))
    d = DevAttn(inp)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = run_attn(d, mode, sms=sms, status=status)
    ref, ref_lse = oracle_attn_full(inp, mode)
    assert_attn_close(out, ref, lse, ref_lse, tag=f"tiny mode={mode} sms={sms}")
    assert status.item() == 0


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("mode", [DRAFT, VERIFY])
@pytest.mark.parametrize("sms", SMS)
def test_shapes(dev, shape, mode, sms):
    name, Hq, Hkv, D, B, ps, lens = shape
    cfg = _cfg(name, len(lens), Hq, Hkv, D, B, ps, lens)
    inp = wl.make_attn_inputs(cfg, extra_pages=2)
    d = DevAttn(inp)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = run_attn(d, mode, sms=sms, status=status)
    ref, ref_lse = oracle_attn_full(inp, mode)
    assert_attn_close(out, ref, lse, ref_lse, tag=f"{name} mode={mode} sms={sms}")
    assert status.item() == 0


def test_unused_slots_hold_nan(dev):
    """Slots past L+B in a request's last page, and unowned pages, never leak into the output."""
    cfg = _cfg("nan_slots", 3, 8, 2, 128, 8, 64, (70, 1, 200))
    inp = wl.make_attn_inputs(cfg, extra_pages=3)
    ps = cfg.page_size
    used = np.zeros(inp.num_pages * ps, bool)
    for r, L in enumerate(inp.seq_lens):
        for t in range(int(L) + cfg.B):
            used[inp.block_table[r, t // ps] * ps + t % ps] = True
    d_clean = DevAttn(inp)
    k_nan, v_nan = inp.k_cache.clone(), inp.v_cache.clone()
    k_nan[torch.from_numpy(~used)] = float("nan")
    v_nan[torch.from_numpy(~used)] = float("nan")
    d_nan = DevAttn(wl.AttnInputs(cfg, inp.seq_lens, inp.block_table, inp.num_pages, inp.q,
                                  k_nan, v_nan, inp.scale))
    for mode in (DRAFT, VERIFY):
        for sms in SMS:
            a, _ = run_attn(d_clean, mode, sms=sms)
            b, _ = run_attn(d_nan, mode, sms=sms)
            assert torch.equal(a, b)


def test_page_permutation_is_bit_identical(dev):
    cfg = _cfg("perm", 2, 16, 4, 128, 16, 32, (900, 333))
    a = wl.make_attn_inputs(cfg, seed=5)
    # same logical sequences, pages shuffled differently in the pool
    rng = np.random.default_rng(99)
    perm = rng.permutation(a.num_pages)
    ps = cfg.page_size
    kp = a.k_cache.view(a.num_pages, ps, cfg.Hkv, cfg.D)
    vp = a.v_cache.view(a.num_pages, ps, cfg.Hkv, cfg.D)
    inv = np.argsort(perm)
    k2 = kp[torch.from_numpy(perm)].reshape_as(a.k_cache).contiguous()
    v2 = vp[torch.from_numpy(perm)].reshape_as(a.v_cache).contiguous()
    table2 = np.where(a.block_table >= 0, inv[np.maximum(a.block_table, 0)], -1).astype(np.int32)
    b = wl.AttnInputs(cfg, a.seq_lens, table2, a.num_pages, a.q, k2, v2, a.scale)
    for mode in (DRAFT, VERIFY):
        for sms in SMS:
            oa, la = run_attn(DevAttn(a), mode, sms=sms)
            ob, lb = run_attn(DevAttn(b), mode, sms=sms)
            assert torch.equal(oa, ob) and torch.equal(la, lb)


def test_mode_relations_are_bit_identical(dev):
    cfg = _cfg("rel", 3, 32, 8, 128, 16, 64, (700, 64, 2000))
    d = DevAttn(wl.make_attn_inputs(cfg))
    od, _ = run_attn(d, DRAFT)
    ov, _ = run_attn(d, VERIFY)
    B = cfg.B
    for r in range(cfg.bs):
        assert torch.equal(od[r * B + B - 1], ov[r * B + B - 1])
    cfg1 = _cfg("b1", 3, 32, 8, 128, 1, 64, (700, 0, 2000))
    d1 = DevAttn(wl.make_attn_inputs(cfg1))
    assert torch.equal(run_attn(d1, DRAFT)[0], run_attn(d1, VERIFY)[0])


def test_bad_page_id_sets_status_and_skips_unit(dev):
    cfg = _cfg("badpage", 3, 8, 2, 128, 8, 16, (100, 200, 50))
    inp = wl.make_attn_inputs(cfg)
    table = inp.block_table.copy()
    table[1, 3] = inp.num_pages + 7  # request 1 references a page outside the pool
    bad = wl.AttnInputs(cfg, inp.seq_lens, table, inp.num_pages, inp.q, inp.k_cache,
                        inp.v_cache, inp.scale)
    d = DevAttn(bad)
    ref, _ = oracle_attn_full(inp, VERIFY)
    # sms = FORCE_SPLIT cuts every unit into one-tile pieces, so only one piece
    # of each of request 1's units sees the bad page and the merge must zero it
    for sms in SMS:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        out, lse = run_attn(d, VERIFY, sms=sms, status=status)
        assert status.item() == 16  # BDSA_DEVICE_OUT_OF_RANGE
        o = out.float().cpu().numpy()
        B = cfg.B
        assert (o[B:2 * B] == 0).all()
        assert (lse[B:2 * B] == float("-inf")).all()
        for r in (0, 2):
            err = np.abs(o[r * B:(r + 1) * B] - ref[r * B:(r + 1) * B])
            assert err.max() < 1e-2


@pytest.mark.parametrize("L_bad", [-1, "beyond_table"])
def test_context_the_table_cannot_hold_sets_status(dev, L_bad):
    # a negative length, or L + B needing more pages than the block-table row
    # holds: the request's rows are zeros (lse -inf), nothing past the row is read
    cfg = _cfg("shapebad", 3, 8, 2, 128, 8, 16, (100, 200, 50))
    inp = wl.make_attn_inputs(cfg)
    ref, _ = oracle_attn_full(inp, VERIFY)
    d = DevAttn(inp)
    max_pages = inp.block_table.shape[1]
    L = -1 if L_bad == -1 else max_pages * cfg.page_size - cfg.B + 1
    d.sl = d.sl.clone()
    d.sl[2] = L
    for sms in SMS:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        out, lse = run_attn(d, VERIFY, sms=sms, status=status)
        assert status.item() == 16
        o = out.float().cpu().numpy()
        B = cfg.B
        assert (o[2 * B:3 * B] == 0).all()
        assert (lse[2 * B:3 * B] == float("-inf")).all()
        err = np.abs(o[:2 * B] - ref[:2 * B])
        assert err.max() < 1e-2


FULL = ["qwen3_8b_verify", "llada2_block_draft", "uno_1k8k_step", "long_ctx_verify"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(dev, name):
    """Full-size workload in the launch configuration the benchmark uses; the oracle
    recomputes sampled requests (first, last, longest, one random)."""
    cfg = wl.config(name)
    inp = wl.make_attn_inputs(cfg, device="cuda")
    d = DevAttn.__new__(DevAttn)
    d.inp, d.q, d.k, d.v = inp, inp.q, inp.k_cache, inp.v_cache
    d.bt = torch.from_numpy(inp.block_table).to(dev)
    d.sl = torch.from_numpy(inp.seq_lens).to(dev)
    rng = np.random.default_rng(3)
    reqs = sorted({0, cfg.bs - 1, int(np.argmax(inp.seq_lens)), int(rng.integers(cfg.bs))})
    if name == "long_ctx_verify":
        reqs = [int(rng.integers(cfg.bs))]
    for mode in cfg.modes:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        out, lse = run_attn(d, mode, status=status)
        assert status.item() == 0
        ref, ref_lse, rows = oracle_attn_requests(d, reqs, mode)
        assert_attn_close(out[torch.from_numpy(rows).to(dev)], ref,
                          lse[torch.from_numpy(rows).to(dev)], ref_lse,
                          tag=f"{name} mode={mode}")
        assert torch.isfinite(out.float()).all()
    del d, inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("sms", [0, FORCE_SPLIT])
def test_output_16_byte_aligned_only(dev, sms):
    """An output buffer that is 16- but not 32-byte aligned (the M = 128 tile
    then stores 16 bytes a lane instead of 32) gives the same bits as an
    aligned one."""
    import block_diffusion_speculative_attn_gb300 as bdsa
    name, Hq, Hkv, D, B, ps, lens = SHAPES[2]  # 128 rows a tile
    cfg = _cfg(name, len(lens), Hq, Hkv, D, B, ps, lens)
    inp = wl.make_attn_inputs(cfg, extra_pages=2)
    d = DevAttn(inp)
    ref, _ = run_attn(d, VERIFY, sms=sms, lse=False)
    n = d.q.numel()
    base = torch.empty(n + 64, dtype=torch.bfloat16, device=dev)
    off = (-(base.data_ptr() // 2) % 16) + 8  # 32-byte boundary + 16 bytes
    out = base[off:off + n].view(d.q.shape)
    assert out.data_ptr() % 32 == 16
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bdsa.block_attn_paged(d.q, d.k, d.v, d.bt, d.sl, B=cfg.B, page_size=cfg.page_size,
                          scale=inp.scale, mode=VERIFY, max_ctx_len=inp.max_ctx_len,
                          num_pages=inp.num_pages, out=out, dev_status=status, sms=sms)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("shape_i,sms", [(2, FORCE_SPLIT), (1, OWNER), (2, OWNER)],
                         ids=["rows128_merge_launch", "rows64_owner_merge",
                              "rows128_owner_merge"])
def test_split_partials_reuse_a_dirty_workspace(dev, shape_i, sms):
    """Split-KV partials are published through ready words in the workspace
    (to the merge launch when the grid is larger than the device, else to the
    owner CTA, for both tiles): calls that reuse one workspace (left by an
    earlier call, or filled with arbitrary bytes) on different inputs each
    match the oracle."""
    import block_diffusion_speculative_attn_gb300 as bdsa
    name, Hq, Hkv, D, B, ps, lens = SHAPES[shape_i]
    ws_bytes = 0
    cases = []
    for seed in (5, 6):
        cfg = _cfg(name, len(lens), Hq, Hkv, D, B, ps, lens, seed=seed)
        inp = wl.make_attn_inputs(cfg, extra_pages=2)
        cases.append((cfg, inp, DevAttn(inp)))
        ws_bytes = max(ws_bytes, bdsa.block_attn_workspace_bytes(
            cfg.bs, cfg.B, cfg.Hq, cfg.Hkv, cfg.D, inp.max_ctx_len, sms))
    ws = torch.randint(0, 256, (ws_bytes,), dtype=torch.uint8, device=dev)
    for rep in range(2):
        for cfg, inp, d in cases:
            status = torch.zeros(1, dtype=torch.int32, device=dev)
            lse = torch.empty((d.q.shape[0], cfg.Hq), dtype=torch.float32, device=dev)
            out = bdsa.block_attn_paged(d.q, d.k, d.v, d.bt, d.sl, B=cfg.B,
                                        page_size=cfg.page_size, scale=inp.scale, mode=VERIFY,
                                        max_ctx_len=inp.max_ctx_len, num_pages=inp.num_pages,
                                        lse=lse, workspace=ws, dev_status=status,
                                        sms=sms)
            torch.cuda.synchronize()
            assert status.item() == 0
            ref, ref_lse = oracle_attn_full(inp, VERIFY)
            assert_attn_close(out, ref, lse, ref_lse, tag=f"reuse {rep} seed {cfg.seed}")


@pytest.mark.parametrize("shape_i,sms", [(2, FORCE_SPLIT), (1, OWNER), (2, OWNER)],
                         ids=["rows128_merge_launch", "rows64_owner_merge",
                              "rows128_owner_merge"])
def test_cuda_graph_replays_with_new_inputs(dev, shape_i, sms):
    """The attention call captured into a CUDA graph (units split, so partials
    and their merge are exercised: by the merge launch for a grid larger than
    the device, by the owner CTA otherwise, whose ready words must not carry
    over from one replay to the next) replays correctly when new inputs are
    copied into the captured buffers between replays."""
    import block_diffusion_speculative_attn_gb300 as bdsa
    name, Hq, Hkv, D, B, ps, lens = SHAPES[shape_i]
    inps = [wl.make_attn_inputs(_cfg(name, len(lens), Hq, Hkv, D, B, ps, lens, seed=s),
                                extra_pages=2) for s in (11, 12, 13)]
    cfg = inps[0].cfg
    d = DevAttn(inps[0])
    q, k, v = d.q.clone(), d.k.clone(), d.v.clone()
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], cfg.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(bdsa.block_attn_workspace_bytes(cfg.bs, cfg.B, cfg.Hq, cfg.Hkv, cfg.D,
                                                     inps[0].max_ctx_len, sms),
                     dtype=torch.uint8, device=dev)

    def call():
        bdsa.block_attn_paged(q, k, v, d.bt, d.sl, B=cfg.B, page_size=cfg.page_size,
                              scale=inps[0].scale, mode=VERIFY, max_ctx_len=inps[0].max_ctx_len,
                              num_pages=inps[0].num_pages, out=out, lse=lse, workspace=ws,
                              sms=sms)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    base = inps[0]
    for other in inps[1:] + inps[:1]:
        # the captured seq_lens and block table with another seed's q, k, v
        inp = wl.AttnInputs(base.cfg, base.seq_lens, base.block_table, base.num_pages,
                            other.q, other.k_cache, other.v_cache, base.scale)
        q.copy_(inp.q)
        k.copy_(inp.k_cache)
        v.copy_(inp.v_cache)
        g.replay()
        torch.cuda.synchronize()
        ref, ref_lse = oracle_attn_full(inp, VERIFY)
        assert_attn_close(out, ref, lse, ref_lse, tag=f"graph replay seed {other.cfg.seed}")
