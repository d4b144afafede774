"""CPU checks of the C-ABI library: it loads, exports every symbol that
include/bdsa.h declares, and its host-side argument checks reject bad calls
synchronously (no call here reaches a CUDA API: each one fails its checks first
or only sizes a workspace for an explicit SM count)."""
import ctypes
import os
import re

import pytest

import block_diffusion_speculative_attn_gb300 as bdsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bdsa.h")


@pytest.fixture(scope="module")
def L():
    from block_diffusion_speculative_attn_gb300 import build
    build.build()
    return bdsa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bdsa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("bdsa_prepare_block", "bdsa_block_attn_paged", "bdsa_spec_accept"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert set(names) == set(bdsa.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    assert L.bdsa_status_string(0) == b"BDSA_OK"
    assert L.bdsa_status_string(16).startswith(b"BDSA_DEVICE_OUT_OF_RANGE")
    assert L.bdsa_status_string(12345) == b"BDSA_UNKNOWN_STATUS"
    assert re.match(rb"^\d+\.\d+\.\d+$", L.bdsa_version())


FAKE = ctypes.c_void_p(0x100000)      # never dereferenced: calls below fail their checks first
FAKE_ODD = ctypes.c_void_p(0x100002)  # 2-byte aligned only


def _attn(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, max_pages=4, num_pages=8, sl=FAKE, max_ctx=100,
             bs=2, B=8, Hq=8, Hkv=2, D=128, ps=16, scale=0.1, mode=1, out=FAKE, lse=None,
             ws=None, ws_bytes=0, sms=152)
    a.update(kw)
    return L.bdsa_block_attn_paged(a["q"], a["k"], a["v"], a["bt"], a["max_pages"],
                                   a["num_pages"], a["sl"], a["max_ctx"], a["bs"], a["B"],
                                   a["Hq"], a["Hkv"], a["D"], a["ps"], a["scale"], a["mode"],
                                   a["out"], a["lse"], a["ws"], a["ws_bytes"], a["sms"], None, None)


def test_attn_host_checks(L):
    assert _attn(L, bs=0) == 0                      # empty batch: nothing to do
    assert _attn(L, q=None) == 1                    # INVALID_ARG
    assert _attn(L, mode=2) == 1
    assert _attn(L, Hq=6, Hkv=4) == 1               # Hq % Hkv
    assert _attn(L, scale=float("nan")) == 1
    assert _attn(L, scale=-0.5) == 1
    assert _attn(L, scale=0.0) == 1
    assert _attn(L, D=96) == 2                      # UNSUPPORTED
    assert _attn(L, B=65) == 2
    assert _attn(L, Hq=64, Hkv=2, B=8) == 2         # G*B = 256 > 128
    assert _attn(L, ps=24) == 2                     # page size not a power of two
    assert _attn(L, ps=4) == 2
    assert _attn(L, q=FAKE_ODD) == 3                # MISALIGNED


def _accept(L, **kw):
    a = dict(ids=FAKE, p=FAKE, psr=16000, psi=1000, q=FAKE, qsr=15000, qsi=1000, ua=FAKE,
             us=FAKE, sl=FAKE, bs=4, B=16, V=1000, outs=FAKE, ws=None, ws_bytes=0, sms=152)
    a.update(kw)
    return L.bdsa_spec_accept(a["ids"], a["p"], a["psr"], a["psi"], a["q"], a["qsr"], a["qsi"],
                              a["ua"], a["us"], a["sl"], a["bs"], a["B"], a["V"], a["outs"],
                              a["outs"], a["outs"], a["outs"], a["outs"], a["ws"], a["ws_bytes"],
                              a["sms"], None, None)


def test_accept_host_checks(L):
    assert _accept(L, bs=0) == 0
    assert _accept(L, p=None) == 1
    assert _accept(L, V=0) == 1
    assert _accept(L, psi=-1) == 1
    assert _accept(L, us=None) == 1                 # stochastic mode needs u_samp
    assert _accept(L, B=65) == 2
    assert _accept(L, p=ctypes.c_void_p(0x100001)) == 3


def test_prepare_host_checks(L):
    f = L.bdsa_prepare_block
    assert f(FAKE, FAKE, FAKE, 4, 8, 0, 8, 16, 0, FAKE, FAKE, FAKE, None, None) == 0
    assert f(None, FAKE, FAKE, 4, 8, 2, 8, 16, 0, FAKE, FAKE, FAKE, None, None) == 1
    assert f(FAKE, FAKE, FAKE, 4, 8, 2, 0, 16, 0, FAKE, FAKE, FAKE, None, None) == 1
    assert f(FAKE, FAKE, FAKE, 4, 8, 2, 8, 0, 0, FAKE, FAKE, FAKE, None, None) == 1


def test_workspace_plans(L):
    # persistent schedule: two partial slots per CTA (bad-page flag, 64-bit
    # ready word, log2-sum-exp per row, output rows)
    def al(x):
        return (x + 255) // 256 * 256
    bs, B, Hq, Hkv, D, sms = 32, 16, 32, 8, 128, 152
    rows = Hq // Hkv * B
    want = (al(2 * sms * 4) + al(2 * sms * 8) + al(2 * sms * rows * 4)
            + al(2 * sms * rows * D * 4))
    assert L.bdsa_block_attn_workspace_bytes(bs, B, Hq, Hkv, D, 4096, sms) == want
    # independent of the context length bound
    assert L.bdsa_block_attn_workspace_bytes(bs, B, Hq, Hkv, D, 131072, sms) == want
    # acceptance: no scratch while a row's segment totals fit one CTA's shared
    # memory (V <= 2^21); beyond that, float-float totals per segment and more
    assert L.bdsa_spec_accept_workspace_bytes(32, 16, 151936, 152) == 0
    assert L.bdsa_spec_accept_workspace_bytes(32, 16, 1 << 21, 152) == 0
    V = (1 << 21) + 1
    assert L.bdsa_spec_accept_workspace_bytes(32, 16, V, 152) > 32 * ((V + 255) // 256) * 8


def _idlm_accept(L, **kw):
    a = dict(ids=FAKE, mode=FAKE, p=FAKE, psr=15000, psi=1000, q=FAKE, qsr=15000, qsi=1000,
             qs=FAKE, ua=FAKE, us=FAKE, sl=FAKE, bs=4, N=8, V=1000, outs=FAKE, ns=FAKE, sms=152)
    a.update(kw)
    o = a["outs"]
    return L.bdsa_idlm_accept(a["ids"], a["mode"], a["p"], a["psr"], a["psi"], a["q"], a["qsr"],
                              a["qsi"], a["qs"], a["ua"], a["us"], a["sl"], a["bs"], a["N"],
                              a["V"], o, o, o, o, o, a["ns"], o, o, o, a["sms"], None, None)


def test_idlm_accept_host_checks(L):
    assert _idlm_accept(L, bs=0) == 0
    assert _idlm_accept(L, bs=-1) == 1
    assert _idlm_accept(L, N=0) == 1
    assert _idlm_accept(L, V=0) == 1
    assert _idlm_accept(L, qsi=-1) == 1
    assert _idlm_accept(L, p=None) == 1
    assert _idlm_accept(L, qs=None) == 1
    assert _idlm_accept(L, q=None) == 1           # N > 1 verifies against q_prev
    assert _idlm_accept(L, ns=None) == 1          # N > 1 draws new specs
    assert _idlm_accept(L, N=33) == 2             # UNSUPPORTED
    assert _idlm_accept(L, V=(1 << 21) + 1) == 2
    assert _idlm_accept(L, p=ctypes.c_void_p(0x100001)) == 3


def test_idlm_prepare_host_checks(L):
    f = L.bdsa_idlm_prepare
    # pending, specs, mode, seq_lens, block_table, max_pages, num_pages, bs, N, ps, mask, outs
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 0, 8, 16, 0, FAKE, FAKE, FAKE, None, None) == 0
    assert f(None, FAKE, FAKE, FAKE, FAKE, 4, 8, 2, 8, 16, 0, FAKE, FAKE, FAKE, None, None) == 1
    assert f(FAKE, None, FAKE, FAKE, FAKE, 4, 8, 2, 8, 16, 0, FAKE, FAKE, FAKE, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 2, 0, 16, 0, FAKE, FAKE, FAKE, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 2, 8, 0, 0, FAKE, FAKE, FAKE, None, None) == 1


def _kvmat(L, **kw):
    a = dict(hidden=FAKE, cl=FAKE, pos=FAKE, loc=FAKE, bs=2, B=16, H=4096, w=FAKE, g=FAKE,
             layers=5, Hkv=8, D=128, cos=FAKE, sin=FAKE, max_pos=8192, eps=1e-6, kc=FAKE,
             vc=FAKE, slots=1 << 20, ws=FAKE, ws_bytes=0)
    a.update(kw)
    return L.bdsa_kv_materialize(a["hidden"], a["cl"], a["pos"], a["loc"], a["bs"], a["B"],
                                 a["H"], a["w"], a["g"], a["layers"], a["Hkv"], a["D"],
                                 a["cos"], a["sin"], a["max_pos"], a["eps"], a["kc"], a["vc"],
                                 a["slots"], a["ws"], a["ws_bytes"], None, None)


def test_kv_materialize_host_checks(L):
    assert _kvmat(L, bs=0) == 0
    assert _kvmat(L, bs=-1) == 1
    assert _kvmat(L, B=0) == 1
    assert _kvmat(L, eps=float("nan")) == 1
    assert _kvmat(L, eps=-1.0) == 1
    assert _kvmat(L, hidden=None) == 1
    assert _kvmat(L, ws=None) == 1
    assert _kvmat(L, D=64) == 2                      # UNSUPPORTED
    assert _kvmat(L, H=4000) == 2
    assert _kvmat(L, hidden=FAKE_ODD) == 3           # MISALIGNED
    assert _kvmat(L, ws_bytes=16) == 4               # WORKSPACE_TOO_SMALL
    # gathered rows: a count, (slot, position) per row, a dense copy of each row
    need = L.bdsa_kv_materialize_workspace_bytes(32, 16, 4096)
    assert need == 256 + 32 * 16 * 8 + 32 * 16 * 4096 * 2


def _tree_attn(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, max_pages=40, num_pages=80, sl=FAKE, max_ctx=100,
             bs=2, B=481, Hq=32, Hkv=8, D=128, ps=16, scale=0.1, mask=FAKE, out=FAKE, lse=None,
             ws=None, ws_bytes=0, sms=152)
    a.update(kw)
    return L.bdsa_block_attn_paged_tree(a["q"], a["k"], a["v"], a["bt"], a["max_pages"],
                                        a["num_pages"], a["sl"], a["max_ctx"], a["bs"], a["B"],
                                        a["Hq"], a["Hkv"], a["D"], a["ps"], a["scale"],
                                        a["mask"], a["out"], a["lse"], a["ws"], a["ws_bytes"],
                                        a["sms"], None, None)


def test_tree_host_checks(L):
    # trees of up to BDSA_TREE_MAX_NODES = 512 nodes (the Psi-Spec Tree
    # sampler's 481), G <= 128: a valid shape gets past the limits to the
    # workspace check
    assert _tree_attn(L) == 4                          # WORKSPACE_TOO_SMALL
    assert _tree_attn(L, B=512) == 4
    assert _tree_attn(L, Hq=256, Hkv=2, B=3) == 4      # G = 128: one node a row tile
    assert _tree_attn(L, B=513) == 2                   # UNSUPPORTED
    assert _tree_attn(L, Hq=258, Hkv=1, B=2) == 2      # G > 128
    assert _tree_attn(L, mask=None) == 1               # INVALID_ARG
    assert _tree_attn(L, mask=ctypes.c_void_p(0x100004)) == 3   # MISALIGNED (8 bytes)
    # the workspace holds partials of 128-row tiles of whole nodes
    def al(x):
        return (x + 255) // 256 * 256
    sms, rows, D = 152, 128, 128
    want = al(2 * sms * 4) + al(2 * sms * 8) + al(2 * sms * rows * 4) + al(2 * sms * rows * D * 4)
    assert L.bdsa_block_attn_workspace_bytes(32, 481, 32, 8, D, 4096, sms) == want
    rows = 42 * 3                                      # G = 3: 42 nodes a tile
    want = al(2 * sms * 4) + al(2 * sms * 8) + al(2 * sms * rows * 4) + al(2 * sms * rows * D * 4)
    assert L.bdsa_block_attn_workspace_bytes(32, 150, 6, 2, D, 4096, sms) == want
    tp = L.bdsa_tree_prepare
    # (empty batches: the size limits are checked before the batch is)
    assert tp(FAKE, FAKE, FAKE, 4, 8, 0, 512, 16, FAKE, FAKE, FAKE, FAKE, None, None) == 0
    assert tp(FAKE, FAKE, FAKE, 4, 8, 0, 513, 16, FAKE, FAKE, FAKE, FAKE, None, None) == 2
    ta = L.bdsa_tree_accept
    o = FAKE
    assert ta(FAKE, FAKE, FAKE, 0, 0, FAKE, FAKE, 0, 512, 1000, o, o, o, o, o, 152, None,
              None) == 0
    assert ta(FAKE, FAKE, FAKE, 0, 0, FAKE, FAKE, 0, 513, 1000, o, o, o, o, o, 152, None,
              None) == 2
