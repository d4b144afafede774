"""Block-diffusion self-speculative draft/verify step for NVIDIA GB300 (sm_103a).

Thin Python binding over the C ABI of ``libbdsa.so`` (declared in
``include/bdsa.h``).  This module only marshals arguments: it checks tensor
dtypes/devices, allocates outputs and workspaces with torch, and passes raw
device pointers plus the current CUDA stream.  Every step of the computation
runs in the library's CUDA kernels; there is no fallback of any kind, and every
call raises if the library is not built or a call returns an error status.

Calls (all asynchronous on the current stream):
  prepare_block     block ids / positions / cache slots of each request's block
  block_attn_paged  block attention over the paged cache, DRAFT or VERIFY mask
  spec_accept       lossless speculative acceptance (stochastic or greedy)
  idlm_prepare      I-DLM Block-N layout of 2N-1 slots (pending, carried specs, masks)
  idlm_accept       I-DLM Block-N verify / correct / draw-new-specs / KV-trim step
  kv_materialize    draft K/V of the committed rows (projection, K norm, RoPE, paged write)
  tree_prepare      token-tree layout: depths, positions, cache slots, ancestor masks
  block_attn_paged(tree_mask=...)  tree attention (block row sees its ancestors)
  tree_accept       lossless tree acceptance walk (stochastic or greedy)
"""
from __future__ import annotations

import ctypes
import os

import torch

DRAFT, VERIFY = 0, 1
_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbdsa.so")

STATUS = {0: "BDSA_OK", 1: "BDSA_INVALID_ARG", 2: "BDSA_UNSUPPORTED", 3: "BDSA_MISALIGNED",
          4: "BDSA_WORKSPACE_TOO_SMALL", 5: "BDSA_CUDA_ERROR", 16: "BDSA_DEVICE_OUT_OF_RANGE",
          17: "BDSA_DEVICE_TIMEOUT"}

# Every symbol include/bdsa.h declares.
EXPORTS = ("bdsa_status_string", "bdsa_version", "bdsa_prepare_block",
           "bdsa_block_attn_workspace_bytes", "bdsa_block_attn_paged",
           "bdsa_block_attn_paged_append", "bdsa_spec_accept_workspace_bytes",
           "bdsa_spec_accept", "bdsa_spec_accept_noalloc", "bdsa_idlm_prepare",
           "bdsa_idlm_accept", "bdsa_kv_materialize_workspace_bytes", "bdsa_kv_materialize",
           "bdsa_tree_prepare", "bdsa_block_attn_paged_tree", "bdsa_tree_accept")

_lib = None


class BdsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


def lib() -> ctypes.CDLL:
    """Load libbdsa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libbdsa.so is not built ({LIB_PATH}); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    L.bdsa_status_string.argtypes = [i32]
    L.bdsa_status_string.restype = ctypes.c_char_p
    L.bdsa_version.argtypes = []
    L.bdsa_version.restype = ctypes.c_char_p
    L.bdsa_prepare_block.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, P]
    L.bdsa_prepare_block.restype = i32
    L.bdsa_block_attn_workspace_bytes.argtypes = [i32] * 7
    L.bdsa_block_attn_workspace_bytes.restype = sz
    L.bdsa_block_attn_paged.argtypes = [P, P, P, P, i32, i32, P, i32, i32, i32, i32, i32, i32,
                                        i32, f32, i32, P, P, P, sz, i32, P, P]
    L.bdsa_block_attn_paged.restype = i32
    L.bdsa_block_attn_paged_append.argtypes = [P, P, P, P, P, P, i32, i32, P, i32, i32, i32, i32,
                                               i32, i32, i32, f32, i32, P, P, P, sz, i32, P, P]
    L.bdsa_block_attn_paged_append.restype = i32
    L.bdsa_spec_accept_workspace_bytes.argtypes = [i32] * 4
    L.bdsa_spec_accept_workspace_bytes.restype = sz
    L.bdsa_spec_accept.argtypes = [P, P, i64, i64, P, i64, i64, P, P, P, i32, i32, i32, P, P, P,
                                   P, P, P, sz, i32, P, P]
    L.bdsa_spec_accept.restype = i32
    L.bdsa_spec_accept_noalloc.argtypes = [P, P, i64, i64, P, i64, i64, P, P, P, i32, i32, i32,
                                           P, P, P, P, P, i32, P, P]
    L.bdsa_spec_accept_noalloc.restype = i32
    L.bdsa_idlm_prepare.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, P]
    L.bdsa_idlm_prepare.restype = i32
    L.bdsa_idlm_accept.argtypes = [P, P, P, i64, i64, P, i64, i64, P, P, P, P, i32, i32, i32,
                                   P, P, P, P, P, P, P, P, P, i32, P, P]
    L.bdsa_idlm_accept.restype = i32
    L.bdsa_kv_materialize_workspace_bytes.argtypes = [i32, i32, i32]
    L.bdsa_kv_materialize_workspace_bytes.restype = sz
    L.bdsa_kv_materialize.argtypes = [P, P, P, P, i32, i32, i32, P, P, i32, i32, i32, P, P, i32,
                                      f32, P, P, i64, P, sz, P, P]
    L.bdsa_kv_materialize.restype = i32
    L.bdsa_tree_prepare.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P]
    L.bdsa_tree_prepare.restype = i32
    L.bdsa_block_attn_paged_tree.argtypes = [P, P, P, P, i32, i32, P, i32, i32, i32, i32, i32,
                                             i32, i32, f32, P, P, P, P, sz, i32, P, P]
    L.bdsa_block_attn_paged_tree.restype = i32
    L.bdsa_tree_accept.argtypes = [P, P, P, i64, i64, P, P, i32, i32, i32, P, P, P, P, P, i32,
                                   P, P]
    L.bdsa_tree_accept.restype = i32
    _lib = L
    return L


def _check(fn: str, status: int):
    if status != 0:
        raise BdsaError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def num_sms(device=None) -> int:
    return torch.cuda.get_device_properties(device).multi_processor_count


# ---------------------------------------------------------------------------
def prepare_block(verified_id, seq_lens, block_table, num_pages: int, B: int, page_size: int,
                  mask_token_id: int, out=None, dev_status=None):
    """bdsa_prepare_block.  Returns (block_ids, positions, cache_loc), int32 [bs, B]."""
    _dev(verified_id, "verified_id", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(block_table, "block_table", torch.int32)
    bs, max_pages = block_table.shape
    if out is None:
        out = tuple(torch.empty((bs, B), dtype=torch.int32, device=block_table.device)
                    for _ in range(3))
    for name, t in zip(("block_ids", "positions", "cache_loc"), out):
        _dev(t, name, torch.int32)
    st = lib().bdsa_prepare_block(_ptr(verified_id), _ptr(seq_lens), _ptr(block_table),
                                  max_pages, num_pages, bs, B, page_size, mask_token_id,
                                  _ptr(out[0]), _ptr(out[1]), _ptr(out[2]), _ptr(dev_status),
                                  _stream(block_table.device))
    _check("bdsa_prepare_block", st)
    return out


def block_attn_workspace_bytes(bs, B, Hq, Hkv, D, max_ctx_len, sms: int = 0) -> int:
    return int(lib().bdsa_block_attn_workspace_bytes(bs, B, Hq, Hkv, D, max_ctx_len, sms))


def block_attn_paged(q, k_cache, v_cache, block_table, seq_lens, *, B: int, page_size: int,
                     scale: float, mode: int, max_ctx_len: int, num_pages: int | None = None,
                     out=None, lse=None, workspace=None, dev_status=None, sms: int = 0,
                     k_new=None, v_new=None, tree_mask=None):
    """bdsa_block_attn_paged.  q [bs*B, Hq, D] bf16, caches [slots, Hkv, D] bf16.

    With k_new / v_new ([bs*B, Hkv, D] bf16) it is bdsa_block_attn_paged_append:
    the block's own keys and values are written into the caches in the same
    launch.  Returns out [bs*B, Hq, D] bf16 (lse is filled when given, fp32
    [bs*B, Hq]).
    """
    _dev(q, "q", torch.bfloat16)
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        _dev(k_new, "k_new", torch.bfloat16)
        _dev(v_new, "v_new", torch.bfloat16)
    _dev(k_cache, "k_cache", torch.bfloat16)
    _dev(v_cache, "v_cache", torch.bfloat16)
    _dev(block_table, "block_table", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    bs, max_pages = block_table.shape
    Hq, D = q.shape[1], q.shape[2]
    Hkv = k_cache.shape[1]
    if num_pages is None:
        num_pages = k_cache.shape[0] // page_size
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", torch.bfloat16)
    if lse is not None:
        _dev(lse, "lse", torch.float32)
    need = block_attn_workspace_bytes(bs, B, Hq, Hkv, D, max_ctx_len, sms)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if tree_mask is not None:
        _dev(tree_mask, "tree_mask", torch.int64)
        if tree_mask.numel() < bs * B * tree_mask_words(B):
            raise ValueError("tree_mask holds fewer than bs * B * ceil(B / 64) words")
        if k_new is not None:
            raise ValueError("the tree call has no fused append")
        st = lib().bdsa_block_attn_paged_tree(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), max_pages, num_pages,
            _ptr(seq_lens), int(max_ctx_len), bs, B, Hq, Hkv, D, page_size, float(scale),
            _ptr(tree_mask), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, sms,
            _ptr(dev_status), _stream(q.device))
        _check("bdsa_block_attn_paged_tree", st)
    elif k_new is None:
        st = lib().bdsa_block_attn_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                         max_pages, num_pages, _ptr(seq_lens), int(max_ctx_len),
                                         bs, B, Hq, Hkv, D, page_size, float(scale), int(mode),
                                         _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, sms,
                                         _ptr(dev_status), _stream(q.device))
        _check("bdsa_block_attn_paged", st)
    else:
        st = lib().bdsa_block_attn_paged_append(
            _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
            max_pages, num_pages, _ptr(seq_lens), int(max_ctx_len), bs, B, Hq, Hkv, D, page_size,
            float(scale), int(mode), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, sms,
            _ptr(dev_status), _stream(q.device))
        _check("bdsa_block_attn_paged_append", st)
    return out


def spec_accept_workspace_bytes(bs, B, V, sms: int = 0) -> int:
    return int(lib().bdsa_spec_accept_workspace_bytes(bs, B, V, sms))


def spec_accept(block_ids, p, q, u_acc, u_samp, seq_lens, *, p_strides=None, q_strides=None,
                V: int | None = None, out=None, workspace=None, dev_status=None, sms: int = 0):
    """bdsa_spec_accept.  q=None selects greedy mode.

    Returns dict with accept_len, commit_len, bonus_id, new_seq_lens ([bs] int32) and
    out_tokens ([bs, B] int32).
    """
    _dev(block_ids, "block_ids", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    if not (p.is_cuda and p.dtype == torch.float32):
        raise TypeError("p must be a CUDA float32 tensor")
    bs, B = block_ids.shape
    V = p.shape[-1] if V is None else V
    if p_strides is None:
        _dev(p, "p", torch.float32)
        p_strides = (B * V, V)
    if q is not None:
        if not (q.is_cuda and q.dtype == torch.float32):
            raise TypeError("q must be a CUDA float32 tensor")
        if q_strides is None:
            _dev(q, "q", torch.float32)
            q_strides = ((B - 1) * V, V)
        _dev(u_acc, "u_acc", torch.float32)
        _dev(u_samp, "u_samp", torch.float32)
    else:
        q_strides = (0, 0)
    dev = block_ids.device
    if out is None:
        out = {k: torch.empty(bs, dtype=torch.int32, device=dev)
               for k in ("accept_len", "commit_len", "bonus_id", "new_seq_lens")}
        out["out_tokens"] = torch.empty((bs, B), dtype=torch.int32, device=dev)
    need = spec_accept_workspace_bytes(bs, B, V, sms)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    # With B == 1 there is no draft and q is never read, but its pointer must stay non-null
    # to select the stochastic rule; an empty tensor may report a null data pointer.
    q_ptr = None if q is None else (_ptr(q) if q.numel() > 0 else _ptr(p))
    st = lib().bdsa_spec_accept(_ptr(block_ids), _ptr(p), int(p_strides[0]), int(p_strides[1]),
                                q_ptr, int(q_strides[0]), int(q_strides[1]),
                                _ptr(u_acc) if q is not None else None,
                                _ptr(u_samp) if q is not None else None, _ptr(seq_lens), bs, B,
                                V, _ptr(out["accept_len"]), _ptr(out["commit_len"]),
                                _ptr(out["out_tokens"]), _ptr(out["bonus_id"]),
                                _ptr(out["new_seq_lens"]), _ptr(workspace), ws_bytes, sms,
                                _ptr(dev_status), _stream(dev))
    _check("bdsa_spec_accept", st)
    return out


# ---------------------------------------------------------------------------
IDLM_KEYS = ("accept_len", "n_out", "next_mode", "next_pending", "next_q_slot",
             "new_seq_lens", "kv_keep")


def idlm_prepare(pending, specs, mode, seq_lens, block_table, num_pages: int, N: int,
                 page_size: int, mask_token_id: int, out=None, dev_status=None):
    """bdsa_idlm_prepare.  specs [bs, N-1] int32 (read in verify mode only).

    Returns (block_ids, positions, cache_loc), int32 [bs, 2N-1].
    """
    _dev(pending, "pending", torch.int32)
    _dev(mode, "mode", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(block_table, "block_table", torch.int32)
    if specs is not None:
        _dev(specs, "specs", torch.int32)
    bs, max_pages = block_table.shape
    blk = 2 * N - 1
    if out is None:
        out = tuple(torch.empty((bs, blk), dtype=torch.int32, device=block_table.device)
                    for _ in range(3))
    for name, t in zip(("block_ids", "positions", "cache_loc"), out):
        _dev(t, name, torch.int32)
    specs_ptr = _ptr(specs) if specs is not None and specs.numel() > 0 else None
    st = lib().bdsa_idlm_prepare(_ptr(pending), specs_ptr, _ptr(mode), _ptr(seq_lens),
                                 _ptr(block_table), max_pages, num_pages, bs, N, page_size,
                                 mask_token_id, _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
                                 _ptr(dev_status), _stream(block_table.device))
    _check("bdsa_idlm_prepare", st)
    return out


def idlm_accept(block_ids, mode, p, q_prev, q_slot, u_acc, u_samp, seq_lens, N: int, *,
                p_strides=None, q_strides=None, V: int | None = None, out=None,
                dev_status=None, sms: int = 0):
    """bdsa_idlm_accept.  p, q_prev fp32 [bs, 2N-1, V] (or addressed through
    the element strides (row, slot)); u_acc [bs, N-1], u_samp [bs, N].

    Returns a dict of int32 tensors: IDLM_KEYS [bs], out_tokens [bs, N] and
    next_specs [bs, N-1].
    """
    _dev(block_ids, "block_ids", torch.int32)
    _dev(mode, "mode", torch.int32)
    _dev(q_slot, "q_slot", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(u_samp, "u_samp", torch.float32)
    bs, blk = block_ids.shape
    if blk != 2 * N - 1:
        raise ValueError(f"block_ids has {blk} slots, want 2N-1 = {2 * N - 1}")
    for name, t in (("p", p), ("q_prev", q_prev)):
        if not (t.is_cuda and t.dtype == torch.float32):
            raise TypeError(f"{name} must be a CUDA float32 tensor")
    V = p.shape[-1] if V is None else V
    if p_strides is None:
        _dev(p, "p", torch.float32)
        p_strides = (blk * V, V)
    if q_strides is None:
        _dev(q_prev, "q_prev", torch.float32)
        q_strides = (blk * V, V)
    if N > 1:
        _dev(u_acc, "u_acc", torch.float32)
    dev = block_ids.device
    if out is None:
        out = {k: torch.empty(bs, dtype=torch.int32, device=dev) for k in IDLM_KEYS}
        out["out_tokens"] = torch.empty((bs, N), dtype=torch.int32, device=dev)
        out["next_specs"] = torch.empty((bs, max(N - 1, 0)), dtype=torch.int32, device=dev)
    ns = out["next_specs"]
    st = lib().bdsa_idlm_accept(
        _ptr(block_ids), _ptr(mode), _ptr(p), int(p_strides[0]), int(p_strides[1]),
        _ptr(q_prev), int(q_strides[0]), int(q_strides[1]), _ptr(q_slot),
        _ptr(u_acc) if N > 1 else None, _ptr(u_samp), _ptr(seq_lens), bs, N, V,
        _ptr(out["accept_len"]), _ptr(out["n_out"]), _ptr(out["out_tokens"]),
        _ptr(out["next_mode"]), _ptr(out["next_pending"]), _ptr(ns) if ns.numel() > 0 else None,
        _ptr(out["next_q_slot"]), _ptr(out["new_seq_lens"]), _ptr(out["kv_keep"]), sms,
        _ptr(dev_status), _stream(dev))
    _check("bdsa_idlm_accept", st)
    return out


# ---------------------------------------------------------------------------
def kv_materialize_workspace_bytes(bs, B, H) -> int:
    return int(lib().bdsa_kv_materialize_workspace_bytes(bs, B, H))


def kv_materialize(hidden, commit_len, positions, cache_loc, w_kv, k_norm_w, rope_cos, rope_sin,
                   k_cache, v_cache, *, B: int, eps: float, workspace=None, dev_status=None):
    """bdsa_kv_materialize: the committed rows' K (RMS norm, RoPE) and V of every
    draft layer, written into k_cache / v_cache [n_layers, slots, Hkv, D] at
    cache_loc.  hidden [bs*B, H] bf16; w_kv [n_layers, 2, Hkv*D, H] bf16;
    k_norm_w [n_layers, D] bf16; rope_cos / rope_sin [max_pos, D/2] fp32."""
    _dev(hidden, "hidden", torch.bfloat16)
    for name, t in (("commit_len", commit_len), ("positions", positions),
                    ("cache_loc", cache_loc)):
        _dev(t, name, torch.int32)
    for name, t in (("w_kv", w_kv), ("k_norm_w", k_norm_w), ("k_cache", k_cache),
                    ("v_cache", v_cache)):
        _dev(t, name, torch.bfloat16)
    _dev(rope_cos, "rope_cos", torch.float32)
    _dev(rope_sin, "rope_sin", torch.float32)
    rows, H = hidden.shape
    bs = commit_len.shape[0]
    if rows != bs * B:
        raise ValueError(f"hidden has {rows} rows, want bs*B = {bs * B}")
    n_layers, _, HD, _ = w_kv.shape
    _, num_slots, Hkv, D = k_cache.shape
    need = kv_materialize_workspace_bytes(bs, B, H)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=hidden.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().bdsa_kv_materialize(
        _ptr(hidden), _ptr(commit_len), _ptr(positions), _ptr(cache_loc), bs, B, H, _ptr(w_kv),
        _ptr(k_norm_w), n_layers, Hkv, D, _ptr(rope_cos), _ptr(rope_sin), rope_cos.shape[0],
        float(eps), _ptr(k_cache), _ptr(v_cache), int(num_slots), _ptr(workspace), ws_bytes,
        _ptr(dev_status), _stream(hidden.device))
    _check("bdsa_kv_materialize", st)


# ---------------------------------------------------------------------------
TREE_KEYS = ("accept_len", "bonus_id", "new_seq_lens")


def tree_mask_words(B: int) -> int:
    """64-bit words of one node's ancestor-or-self set in a tree of B nodes."""
    return (B + 63) // 64


def tree_prepare(parent, seq_lens, block_table, num_pages: int, page_size: int, out=None,
                 dev_status=None):
    """bdsa_tree_prepare.  parent [bs, B] int32 (node 0 the root, parent -1).
    Returns (depth, positions, cache_loc) int32 [bs, B] and tree_mask int64
    [bs, B, ceil(B / 64)] (uint64 words of ancestor-or-self bits)."""
    _dev(parent, "parent", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(block_table, "block_table", torch.int32)
    bs, B = parent.shape
    dev = parent.device
    if out is None:
        out = tuple(torch.empty((bs, B), dtype=torch.int32, device=dev) for _ in range(3)) + \
            (torch.empty((bs, B, tree_mask_words(B)), dtype=torch.int64, device=dev),)
    if out[3].numel() < bs * B * tree_mask_words(B):
        raise ValueError("tree_mask holds fewer than bs * B * ceil(B / 64) words")
    st = lib().bdsa_tree_prepare(_ptr(parent), _ptr(seq_lens), _ptr(block_table),
                                 block_table.shape[1], num_pages, bs, B, page_size, _ptr(out[0]),
                                 _ptr(out[1]), _ptr(out[2]), _ptr(out[3]), _ptr(dev_status),
                                 _stream(dev))
    _check("bdsa_tree_prepare", st)
    return out


def tree_accept(block_ids, parent, p, u, seq_lens, *, p_strides=None, V: int | None = None,
                out=None, dev_status=None, sms: int = 0):
    """bdsa_tree_accept (u None: greedy).  p fp32 [bs, B, V].  Returns a dict:
    TREE_KEYS [bs], path [bs, B], out_tokens [bs, B] (int32)."""
    _dev(block_ids, "block_ids", torch.int32)
    _dev(parent, "parent", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    if not (p.is_cuda and p.dtype == torch.float32):
        raise TypeError("p must be a CUDA float32 tensor")
    bs, B = block_ids.shape
    V = p.shape[-1] if V is None else V
    if p_strides is None:
        _dev(p, "p", torch.float32)
        p_strides = (B * V, V)
    if u is not None:
        _dev(u, "u", torch.float32)
    dev = block_ids.device
    if out is None:
        out = {k: torch.empty(bs, dtype=torch.int32, device=dev) for k in TREE_KEYS}
        out["path"] = torch.empty((bs, B), dtype=torch.int32, device=dev)
        out["out_tokens"] = torch.empty((bs, B), dtype=torch.int32, device=dev)
    st = lib().bdsa_tree_accept(_ptr(block_ids), _ptr(parent), _ptr(p), int(p_strides[0]),
                                int(p_strides[1]), _ptr(u), _ptr(seq_lens), bs, B, V,
                                _ptr(out["accept_len"]), _ptr(out["path"]),
                                _ptr(out["out_tokens"]), _ptr(out["bonus_id"]),
                                _ptr(out["new_seq_lens"]), sms, _ptr(dev_status), _stream(dev))
    _check("bdsa_tree_accept", st)
    return out
