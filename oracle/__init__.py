"""fp64 CPU oracle for the block-diffusion draft/verify step (test infrastructure).

This package is the checker, not the product.  Only ``tests/``, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` import it.  The
CUDA library never links or calls it, and it shares no code with the library:
the arithmetic lives in ``bdsa_oracle.c`` (plain C, fp64), written from the
source pages' definitions:

* prepare block -- "From DFlash to dLLM Self-Spec (II): SGLang Spec V2",
  section 2.2.2; "... (IV)", section 4.4.1 (block init).
* block attention masks -- "SGLang dLLM / LLaDA 2.0", section "Attention Mask";
  "... (IV)", section 4.4.1 (causal verify over the past KV).
* the block's own K/V appended to the paged cache -- "... (II)", sections 2.2.2
  and 2.2.4 (numpy indexing in this module).
* I-DLM Block-N round -- "... (IV)", sections 4.3 and 4.3.1 (2N-1 layout,
  verify of the carried specs, correction / bonus, new specs from the MASK
  slots) and 4.6 (KV trim, the request's advance).
* KV materialisation of the committed prefix -- "... (II)", section 2.2.6 and
  the DFlash engineering notes (projection across draft layers, K RMS norm,
  rotate-half RoPE from a cos / sin table, write at the verify cache slots).
* tree verify -- "Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
  the Psi-Spec Tree sampler (a token tree verified in parallel with tree
  attention, lossless rejection sampling); "SGLang dLLM / LLaDA 2.0",
  "Attention Mask" (the intra-block mask follows the verify structure).
* acceptance -- "... (IV)", section 4.3.1 (min(1, p/q), correction token);
  "Unlocking Lossless Speedups in LLMs via Discrete Diffusion", background on
  speculative decoding and the Psi-Spec step (longest accepted prefix, residual
  resampling, first token always accepted); "... (II)", section 2.2.5 (greedy
  accept/bonus, commit_len = accept_len + 1).

Pins (tests/test_oracle_*.py): torch CPU scaled_dot_product_attention in fp64
(causal prefill / unmasked / decode special cases), closed forms (constant V,
zero Q with lse = log n), page-permutation invariance, hand-worked acceptance
fixtures under tests/golden/, numpy searchsorted for the sampling rule, and the
lossless property by chi-square and the 1 - TV acceptance rate.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bdsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile bdsa_oracle.c into liboracle.so (gcc, -O2, OpenMP, strict fp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_prepare_block.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, P, P, P]
        lib.oracle_prepare_block.restype = i32
        lib.oracle_block_attn.argtypes = [P, P, P, P, i32, i32, P, i32, i32, i32, i32, i32,
                                          i32, f64, i32, P, P, i32]
        lib.oracle_block_attn.restype = i32
        lib.oracle_spec_accept.argtypes = [P, P, i64, i64, P, i64, i64, P, P, P, i32, i32, i32,
                                           P, P, P, P, P, P, i32]
        lib.oracle_spec_accept.restype = None
        lib.oracle_idlm_prepare.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, P,
                                            P]
        lib.oracle_idlm_prepare.restype = i32
        lib.oracle_idlm_accept.argtypes = [P, P, P, i64, i64, P, i64, i64, P, P, P, P, i32, i32,
                                           i32, P, P, P, P, P, P, P, P, P, P, i32]
        lib.oracle_idlm_accept.restype = None
        lib.oracle_kv_materialize.argtypes = [P, P, P, P, P, P, P, P, i32, f64, i32, i32, i32,
                                               i32, i32, i32, i64, P, P, P, i32]
        lib.oracle_kv_materialize.restype = i32
        lib.oracle_tree_prepare.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P, P, i32]
        lib.oracle_tree_prepare.restype = i32
        lib.oracle_block_attn_tree.argtypes = [P, P, P, P, i32, i32, P, P, i32, i32, i32, i32,
                                               i32, i32, f64, P, P, i32]
        lib.oracle_block_attn_tree.restype = i32
        lib.oracle_tree_accept.argtypes = [P, P, P, i64, i64, P, P, i32, i32, i32, P, P, P, P, P,
                                           P, i32]
        lib.oracle_tree_accept.restype = None
        lib.oracle_inv_cdf.argtypes = [P, i32, f64, P]
        lib.oracle_inv_cdf.restype = i32
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def prepare_block(verified_id, seq_lens, block_table, num_pages, B, page_size, mask_token_id):
    """Returns (block_ids, positions, cache_loc, n_out_of_range), each [bs, B] int32."""
    lib = _load()
    verified_id = _c(verified_id, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    block_table = _c(block_table, np.int32)
    bs, max_pages = block_table.shape
    block_ids = np.empty((bs, B), np.int32)
    positions = np.empty((bs, B), np.int32)
    cache_loc = np.empty((bs, B), np.int32)
    bad = lib.oracle_prepare_block(_ptr(verified_id), _ptr(seq_lens), _ptr(block_table),
                                   max_pages, num_pages, bs, B, page_size, mask_token_id,
                                   _ptr(block_ids), _ptr(positions), _ptr(cache_loc))
    return block_ids, positions, cache_loc, int(bad)


def block_attn(q_bits, k_bits, v_bits, block_table, seq_lens, B, Hq, Hkv, D, page_size,
               scale, mode, num_pages=None, nthreads=1):
    """fp64 block attention.

    q_bits: uint16 bf16 bit patterns [bs*B, Hq, D]; k_bits/v_bits: [slots, Hkv, D].
    mode: 0 = DRAFT (bidirectional block), 1 = VERIFY (token-causal block).
    Returns (out [bs*B, Hq, D] fp64, lse [bs*B, Hq] fp64 natural log).
    """
    lib = _load()
    q_bits = _c(q_bits, np.uint16)
    k_bits = _c(k_bits, np.uint16)
    v_bits = _c(v_bits, np.uint16)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    bs, max_pages = block_table.shape
    if num_pages is None:
        num_pages = k_bits.shape[0] // page_size
    out = np.empty((bs * B, Hq, D), np.float64)
    lse = np.empty((bs * B, Hq), np.float64)
    bad = lib.oracle_block_attn(_ptr(q_bits), _ptr(k_bits), _ptr(v_bits), _ptr(block_table),
                                max_pages, num_pages, _ptr(seq_lens), bs, B, Hq, Hkv, D,
                                page_size, float(scale), int(mode), _ptr(out), _ptr(lse),
                                int(nthreads))
    if bad:
        raise ValueError(f"oracle: {bad} rows referenced out-of-range pages")
    return out, lse


def append_block_kv(k_bits, v_bits, k_new_bits, v_new_bits, block_table, seq_lens, B, page_size,
                    num_pages=None):
    """The block's own keys and values written into copies of the caches.

    "From DFlash to dLLM Self-Spec (II)", sections 2.2.2 and 2.2.4: row r*B + i of
    k_new / v_new ([bs*B, Hkv, D]) is position L_r + i of request r and goes to
    slot block_table[r, (L_r+i) // ps] * ps + (L_r+i) % ps of every KV head.  A
    position whose page is past the block-table row or outside [0, num_pages) is
    not written, nor is any position of a request with L_r < 0.
    Returns (k_bits', v_bits') as new arrays.
    """
    k_out = np.array(k_bits, copy=True)
    v_out = np.array(v_bits, copy=True)
    bt = np.asarray(block_table)
    sl = np.asarray(seq_lens)
    bs, max_pages = bt.shape
    if num_pages is None:
        num_pages = k_out.shape[0] // page_size
    for r in range(bs):
        L = int(sl[r])
        if L < 0:
            continue
        for i in range(B):
            t = L + i
            page = t // page_size
            if page >= max_pages:
                continue
            pg = int(bt[r, page])
            if pg < 0 or pg >= num_pages:
                continue
            slot = pg * page_size + t % page_size
            k_out[slot] = k_new_bits[r * B + i]
            v_out[slot] = v_new_bits[r * B + i]
    return k_out, v_out


def spec_accept(block_ids, p, q, u_acc, u_samp, seq_lens, *, p_strides=None, q_strides=None,
                V=None, nthreads=1):
    """Speculative acceptance (stochastic if q is not None, else greedy).

    p: fp32 [bs, B, V] (or any array addressed through p_strides=(stride_r, stride_i)),
    q: fp32 [bs, B-1, V] or None.  Returns dict of int32 arrays and 'flags'.
    """
    lib = _load()
    block_ids = _c(block_ids, np.int32)
    bs, B = block_ids.shape
    p = np.ascontiguousarray(p, dtype=np.float32)
    if V is None:
        V = p.shape[-1]
    if p_strides is None:
        p_strides = (B * V, V)
    if q is not None:
        q = np.ascontiguousarray(q, dtype=np.float32)
        if q_strides is None:
            q_strides = ((B - 1) * V, V)
    else:
        q_strides = (0, 0)
    u_acc = _c(u_acc, np.float32)
    u_samp = _c(u_samp, np.float32)
    seq_lens = _c(seq_lens, np.int32)
    out = {k: np.empty(bs, np.int32) for k in ("accept_len", "commit_len", "bonus_id",
                                                "new_seq_lens", "flags")}
    out["out_tokens"] = np.empty((bs, B), np.int32)
    lib.oracle_spec_accept(_ptr(block_ids), _ptr(p), p_strides[0], p_strides[1], _ptr(q),
                           q_strides[0], q_strides[1], _ptr(u_acc), _ptr(u_samp),
                           _ptr(seq_lens), bs, B, V, _ptr(out["accept_len"]),
                           _ptr(out["commit_len"]), _ptr(out["out_tokens"]),
                           _ptr(out["bonus_id"]), _ptr(out["new_seq_lens"]), _ptr(out["flags"]),
                           int(nthreads))
    return out


def idlm_prepare(pending, specs, mode, seq_lens, block_table, num_pages, N, page_size,
                 mask_token_id):
    """I-DLM Block-N layout of 2N-1 slots.  specs: [bs, N-1] (read in verify
    mode only).  Returns (block_ids, positions, cache_loc, n_out_of_range)."""
    lib = _load()
    pending = _c(pending, np.int32)
    mode = _c(mode, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    block_table = _c(block_table, np.int32)
    bs, max_pages = block_table.shape
    specs = _c(specs, np.int32).reshape(bs, max(N - 1, 0))
    blk = 2 * N - 1
    out = [np.empty((bs, blk), np.int32) for _ in range(3)]
    bad = lib.oracle_idlm_prepare(_ptr(pending), _ptr(specs), _ptr(mode), _ptr(seq_lens),
                                  _ptr(block_table), max_pages, num_pages, bs, N, page_size,
                                  mask_token_id, *[_ptr(o) for o in out])
    return out[0], out[1], out[2], int(bad)


IDLM_KEYS = ("accept_len", "n_out", "next_mode", "next_pending", "next_q_slot",
             "new_seq_lens", "kv_keep")


def idlm_accept(block_ids, mode, p, q_prev, q_slot, u_acc, u_samp, seq_lens, N, *,
                p_strides=None, q_strides=None, V=None, nthreads=1):
    """I-DLM verify / sample / trim step.  p, q_prev: fp32 [bs, 2N-1, V] (or
    addressed through the strides); u_acc [bs, N-1], u_samp [bs, N].  Returns
    a dict of int32 arrays: IDLM_KEYS [bs], out_tokens [bs, N], next_specs
    [bs, N-1], flags [bs]."""
    lib = _load()
    block_ids = _c(block_ids, np.int32)
    bs, blk = block_ids.shape
    assert blk == 2 * N - 1
    p = np.ascontiguousarray(p, dtype=np.float32)
    q_prev = np.ascontiguousarray(q_prev, dtype=np.float32)
    if V is None:
        V = p.shape[-1]
    if p_strides is None:
        p_strides = (blk * V, V)
    if q_strides is None:
        q_strides = (blk * V, V)
    out = {k: np.empty(bs, np.int32) for k in IDLM_KEYS + ("flags",)}
    out["out_tokens"] = np.empty((bs, N), np.int32)
    out["next_specs"] = np.empty((bs, max(N - 1, 0)), np.int32)
    lib.oracle_idlm_accept(_ptr(block_ids), _ptr(_c(mode, np.int32)), _ptr(p), p_strides[0],
                           p_strides[1], _ptr(q_prev), q_strides[0], q_strides[1],
                           _ptr(_c(q_slot, np.int32)), _ptr(_c(u_acc, np.float32)),
                           _ptr(_c(u_samp, np.float32)), _ptr(_c(seq_lens, np.int32)), bs, N, V,
                           _ptr(out["accept_len"]), _ptr(out["n_out"]), _ptr(out["out_tokens"]),
                           _ptr(out["next_mode"]), _ptr(out["next_pending"]),
                           _ptr(out["next_specs"]), _ptr(out["next_q_slot"]),
                           _ptr(out["new_seq_lens"]), _ptr(out["kv_keep"]), _ptr(out["flags"]),
                           int(nthreads))
    return out


def inv_cdf(w, u):
    """InvCDF(w, u): smallest k with C_k > u*S (fp64 sums).  Returns (k, near_flag)."""
    lib = _load()
    w = _c(w, np.float32)
    flag = np.zeros(1, np.int32)
    k = lib.oracle_inv_cdf(_ptr(w), w.shape[0], float(u), _ptr(flag))
    return int(k), bool(flag[0])


def kv_materialize(hidden_bits, commit_len, positions, cache_loc, w_bits, k_norm_bits, cos_tab,
                   sin_tab, eps, B, n_layers, Hkv, D, num_slots, nthreads=1):
    """fp64 K/V of the committed rows.

    hidden_bits [bs*B, H] and w_bits [n_layers, 2, Hkv*D, H], k_norm_bits
    [n_layers, D]: uint16 bf16 bit patterns; cos_tab / sin_tab [max_pos, D/2]
    fp32.  Returns (k [bs*B, n_layers, Hkv, D] fp64, v (same), status [bs*B]
    int32: 1 written, 0 not committed, -1 skipped for a bad slot / position);
    rows not written hold NaN.
    """
    lib = _load()
    hidden_bits = _c(hidden_bits, np.uint16)
    rows, H = hidden_bits.shape
    bs = rows // B
    w_bits = _c(w_bits, np.uint16)
    assert w_bits.size == n_layers * 2 * Hkv * D * H
    k_norm_bits = _c(k_norm_bits, np.uint16)
    cos_tab = _c(cos_tab, np.float32)
    sin_tab = _c(sin_tab, np.float32)
    max_pos = cos_tab.shape[0]
    k = np.full((rows, n_layers, Hkv, D), np.nan)
    v = np.full((rows, n_layers, Hkv, D), np.nan)
    status = np.empty(rows, np.int32)
    lib.oracle_kv_materialize(_ptr(hidden_bits), _ptr(_c(commit_len, np.int32)),
                              _ptr(_c(positions, np.int32)), _ptr(_c(cache_loc, np.int32)),
                              _ptr(w_bits), _ptr(k_norm_bits), _ptr(cos_tab), _ptr(sin_tab),
                              max_pos, float(eps), bs, B, H, n_layers, Hkv, D, int(num_slots),
                              _ptr(k), _ptr(v), _ptr(status), int(nthreads))
    return k, v, status


def tree_prepare(parent, seq_lens, block_table, num_pages, page_size):
    """Token tree of B nodes per request (parent [bs, B], node 0 the root with
    parent -1).  Returns (depth, positions, cache_loc [bs, B] int32, mask
    [bs, B, ceil(B / 64)] uint64: bit j % 64 of word j // 64 set iff node j is
    the node or one of its ancestors, n_bad)."""
    lib = _load()
    parent = _c(parent, np.int32)
    bs, B = parent.shape
    block_table = _c(block_table, np.int32)
    out = [np.empty((bs, B), np.int32) for _ in range(3)]
    W = (B + 63) // 64
    mask = np.empty((bs, B, W), np.uint64)
    bad = lib.oracle_tree_prepare(_ptr(parent), _ptr(_c(seq_lens, np.int32)), _ptr(block_table),
                                  block_table.shape[1], num_pages, bs, B, page_size,
                                  *[_ptr(o) for o in out], _ptr(mask), W)
    return out[0], out[1], out[2], mask, int(bad)


def block_attn_tree(q_bits, k_bits, v_bits, block_table, seq_lens, parent, B, Hq, Hkv, D,
                    page_size, scale, num_pages=None, nthreads=1):
    """fp64 tree attention: block row i sees the context and its ancestors-or-self."""
    lib = _load()
    q_bits = _c(q_bits, np.uint16)
    k_bits = _c(k_bits, np.uint16)
    v_bits = _c(v_bits, np.uint16)
    block_table = _c(block_table, np.int32)
    bs, max_pages = block_table.shape
    if num_pages is None:
        num_pages = k_bits.shape[0] // page_size
    out = np.empty((bs * B, Hq, D), np.float64)
    lse = np.empty((bs * B, Hq), np.float64)
    bad = lib.oracle_block_attn_tree(_ptr(q_bits), _ptr(k_bits), _ptr(v_bits), _ptr(block_table),
                                     max_pages, num_pages, _ptr(_c(seq_lens, np.int32)),
                                     _ptr(_c(parent, np.int32)), bs, B, Hq, Hkv, D, page_size,
                                     float(scale), _ptr(out), _ptr(lse), int(nthreads))
    if bad:
        raise ValueError(f"oracle: {bad} rows referenced out-of-range pages")
    return out, lse


TREE_KEYS = ("accept_len", "bonus_id", "new_seq_lens")


def tree_accept(block_ids, parent, p, u, seq_lens, *, p_strides=None, V=None, nthreads=1):
    """Tree acceptance (u None: greedy).  p: fp32 [bs, B, V].  Returns a dict of
    int32 arrays: TREE_KEYS [bs], path [bs, B], out_tokens [bs, B], flags [bs]."""
    lib = _load()
    block_ids = _c(block_ids, np.int32)
    bs, B = block_ids.shape
    p = np.ascontiguousarray(p, dtype=np.float32)
    if V is None:
        V = p.shape[-1]
    if p_strides is None:
        p_strides = (B * V, V)
    out = {k: np.empty(bs, np.int32) for k in TREE_KEYS + ("flags",)}
    out["path"] = np.empty((bs, B), np.int32)
    out["out_tokens"] = np.empty((bs, B), np.int32)
    lib.oracle_tree_accept(_ptr(block_ids), _ptr(_c(parent, np.int32)), _ptr(p), p_strides[0],
                           p_strides[1], None if u is None else _ptr(_c(u, np.float32)),
                           _ptr(_c(seq_lens, np.int32)), bs, B, V, _ptr(out["accept_len"]),
                           _ptr(out["path"]), _ptr(out["out_tokens"]), _ptr(out["bonus_id"]),
                           _ptr(out["new_seq_lens"]), _ptr(out["flags"]), int(nthreads))
    return out
