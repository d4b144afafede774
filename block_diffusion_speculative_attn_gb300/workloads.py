"""Seeded synthetic workloads for the draft/verify step.

This module only draws random inputs with the shapes, value distributions and
paging structure of the source pages' workloads; it holds none of the step's
arithmetic (no attention, no acceptance rule, no block layout).  Both the CUDA
path and the CPU oracle consume what it returns.

Structure (sequence lengths, page permutation, block tables) comes from numpy
PCG64; large tensors come from a seeded torch generator on the requested device
so that multi-GB caches are drawn where they live.  bf16 values are fp32
N(0, 1) rounded to nearest even.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

DRAFT, VERIFY = 0, 1


@dataclasses.dataclass(frozen=True)
class StepConfig:
    """One synthetic workload.  ctx is (lo, hi) inclusive, or a tuple of exact lengths."""
    name: str
    bs: int
    Hq: int
    Hkv: int
    D: int
    B: int
    page_size: int
    ctx: tuple
    modes: tuple               # attention passes in step order, DRAFT=0 / VERIFY=1
    V: int = 0                 # 0: no acceptance stage
    accept: str = ""           # "indep2" | "perturb" | "near_uniform" | ""
    seed: int = 1234

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def mask_token_id(self) -> int:
        return max(self.V - 1, 0)


# The five workloads, index order fixed (seed = 1234 + index).
CONFIGS = {
    # Tiny case: 2 requests, GQA 2/1, D 64, contexts 200 and 256, 16-token pages
    # shuffled in the pool, B = 8, both modes; acceptance over a 1000-token vocab.
    "tiny": StepConfig("tiny", 2, 2, 1, 64, 8, 16, (200, 256), (DRAFT, VERIFY), 1000, "indep2",
                       1234),
    # Qwen3-8B-shaped DFlash verify: 32 requests, 32/8 heads, D 128, contexts U[1024, 4096],
    # 64-token pages, B = 16 causal; acceptance over 151936 tokens, q = p with logit noise.
    "qwen3_8b_verify": StepConfig("qwen3_8b_verify", 32, 32, 8, 128, 16, 64, ((1024, 4096),),
                                  (VERIFY,), 151936, "perturb", 1235),
    # LLaDA2.0-style block diffusion draft: 64 requests, 16/4 heads, B = 32 bidirectional,
    # contexts U[512, 8192], 32-token pages, no acceptance stage.
    "llada2_block_draft": StepConfig("llada2_block_draft", 64, 16, 4, 128, 32, 32,
                                     ((512, 8192),), (DRAFT,), 0, "", 1236),
    # Uno 1K/8K-shaped high-concurrency step: 256 requests, 32/8 heads, contexts
    # U[1024, 9216], B = 16: draft pass then verify pass on the same cache, then acceptance.
    "uno_1k8k_step": StepConfig("uno_1k8k_step", 256, 32, 8, 128, 16, 64, ((1024, 9216),),
                                (DRAFT, VERIFY), 151936, "perturb", 1237),
    # Long context, low batch: 4 requests of 131072 tokens, 64/8 heads, B = 16 causal,
    # split-KV path; acceptance with near-uniform q (high rejection).
    "long_ctx_verify": StepConfig("long_ctx_verify", 4, 64, 8, 128, 16, 64, (131072,) * 4,
                                  (VERIFY,), 151936, "near_uniform", 1238),
}
CONFIG_ORDER = list(CONFIGS)


def config(name: str) -> StepConfig:
    return CONFIGS[name]


# ---------------------------------------------------------------------------
# Structure: sequence lengths, page pool permutation, block tables (numpy).

def seq_lens_for(cfg: StepConfig, rng: np.random.Generator) -> np.ndarray:
    if len(cfg.ctx) == 1 and isinstance(cfg.ctx[0], tuple):
        lo, hi = cfg.ctx[0]
        return rng.integers(lo, hi + 1, size=cfg.bs, dtype=np.int64).astype(np.int32)
    assert len(cfg.ctx) == cfg.bs
    return np.asarray(cfg.ctx, dtype=np.int32)


def paging_for(seq_lens: np.ndarray, B: int, page_size: int, rng: np.random.Generator,
               extra_pages: int = 0, max_pages_per_req: int | None = None):
    """Each request owns ceil((L+B)/ps) pages drawn from a randomly permuted pool.

    Returns (block_table [bs, max_pages] int32 with -1 past the owned pages, num_pages).
    """
    need = [(int(L) + B + page_size - 1) // page_size for L in seq_lens]
    total = sum(need) + extra_pages
    perm = rng.permutation(total).astype(np.int32)
    max_pages = max(need) if max_pages_per_req is None else max_pages_per_req
    table = np.full((len(seq_lens), max_pages), -1, dtype=np.int32)
    at = 0
    for r, n in enumerate(need):
        table[r, :n] = perm[at:at + n]
        at += n
    return table, total


@dataclasses.dataclass
class AttnInputs:
    cfg: StepConfig
    seq_lens: np.ndarray        # [bs] int32, committed context length L_r
    block_table: np.ndarray     # [bs, max_pages] int32
    num_pages: int
    q: torch.Tensor             # [bs*B, Hq, D] bf16
    k_cache: torch.Tensor       # [num_pages*ps, Hkv, D] bf16
    v_cache: torch.Tensor       # [num_pages*ps, Hkv, D] bf16
    scale: float

    @property
    def max_ctx_len(self) -> int:
        return int(self.seq_lens.max())


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, g: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_attn_inputs(cfg: StepConfig, device="cpu", seed: int | None = None,
                     seq_lens: np.ndarray | None = None, extra_pages: int = 0) -> AttnInputs:
    seed = cfg.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    if seq_lens is None:
        seq_lens = seq_lens_for(cfg, rng)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    table, num_pages = paging_for(seq_lens, cfg.B, cfg.page_size, rng, extra_pages)
    g = _gen(device, seed)
    slots = num_pages * cfg.page_size
    q = randn_bf16((cfg.bs * cfg.B, cfg.Hq, cfg.D), g, device)
    k = randn_bf16((slots, cfg.Hkv, cfg.D), g, device)
    v = randn_bf16((slots, cfg.Hkv, cfg.D), g, device)
    return AttnInputs(cfg, seq_lens, table, num_pages, q, k, v, 1.0 / math.sqrt(cfg.D))


# ---------------------------------------------------------------------------
# Acceptance inputs: verifier p, draft q, drafts sampled from q, uniforms.

@dataclasses.dataclass
class AcceptInputs:
    block_ids: torch.Tensor     # [bs, B] int32: verified token, then drafts d_1..d_{B-1}
    p: torch.Tensor             # [bs, B, V] fp32
    q: torch.Tensor             # [bs, B-1, V] fp32
    u_acc: torch.Tensor         # [bs, B-1] fp32 in [0, 1)
    u_samp: torch.Tensor        # [bs] fp32 in [0, 1)
    seq_lens: torch.Tensor      # [bs] int32


def make_accept_inputs(cfg: StepConfig, device="cpu", seed: int | None = None,
                       bs: int | None = None, seq_lens: np.ndarray | None = None) -> AcceptInputs:
    seed = (cfg.seed if seed is None else seed) + 7919
    bs = cfg.bs if bs is None else bs
    B, V = cfg.B, cfg.V
    g = _gen(device, seed)
    f32 = torch.float32
    if cfg.accept == "indep2":
        p = torch.softmax(2.0 * torch.randn((bs, B, V), generator=g, device=device, dtype=f32), -1)
        q = torch.softmax(2.0 * torch.randn((bs, B - 1, V), generator=g, device=device,
                                            dtype=f32), -1)
    elif cfg.accept == "perturb":
        logits = 3.0 * torch.randn((bs, B, V), generator=g, device=device, dtype=f32)
        p = torch.softmax(logits, -1)
        noise = torch.randn((bs, B - 1, V), generator=g, device=device, dtype=f32)
        q = torch.softmax(logits[:, :B - 1] + noise, -1)
        del logits, noise
    elif cfg.accept == "near_uniform":
        p = torch.softmax(3.0 * torch.randn((bs, B, V), generator=g, device=device, dtype=f32), -1)
        q = torch.softmax(0.1 * torch.randn((bs, B - 1, V), generator=g, device=device,
                                            dtype=f32), -1)
    else:
        raise ValueError(f"config {cfg.name} has no acceptance stage")
    drafts = torch.multinomial(q.reshape(-1, V), 1, generator=g).reshape(bs, B - 1)
    verified = torch.randint(0, V, (bs, 1), generator=g, device=device)
    block_ids = torch.cat([verified, drafts], dim=1).to(torch.int32).contiguous()
    u_acc = torch.rand((bs, B - 1), generator=g, device=device, dtype=f32)
    u_samp = torch.rand((bs,), generator=g, device=device, dtype=f32)
    if seq_lens is None:
        seq_lens = torch.randint(1, 4096, (bs,), generator=g, device=device).to(torch.int32)
    else:
        seq_lens = torch.as_tensor(np.asarray(seq_lens, np.int32), device=device)
    return AcceptInputs(block_ids, p.contiguous(), q.contiguous(), u_acc, u_samp, seq_lens)


@dataclasses.dataclass
class IdlmInputs:
    """Inputs of one I-DLM Block-N round (blk = 2N - 1 slots per request)."""
    N: int
    pending: torch.Tensor       # [bs] int32, the token whose KV the round writes first
    specs: torch.Tensor         # [bs, N-1] int32, carried specs (meaningful where mode == 1)
    mode: torch.Tensor          # [bs] int32, 1 verify / 0 cold start
    q_slot: torch.Tensor        # [bs] int32, q_prev row of spec_0
    p: torch.Tensor             # [bs, blk, V] fp32, this round's distributions
    q_prev: torch.Tensor        # [bs, blk, V] fp32, the previous round's distributions
    u_acc: torch.Tensor         # [bs, N-1] fp32
    u_samp: torch.Tensor        # [bs, N] fp32
    seq_lens: torch.Tensor      # [bs] int32


def make_idlm_inputs(cfg: StepConfig, N: int = 8, device="cpu", seed: int | None = None,
                     bs: int | None = None, verify_frac: float = 0.75) -> IdlmInputs:
    """A round shaped like cfg's acceptance stage: p = softmax(3 N(0,1) logits);
    the previous round's rows that drew the carried specs are p's logits plus
    N(0,1) noise (the draft is close to the verifier), the other q_prev rows
    independent; a verify_frac share of requests verify carried specs, drawn
    from their q_prev rows at q_slot in {1, N} (after a cold start or after a
    fully verified round); the rest start cold."""
    seed = (cfg.seed if seed is None else seed) + 104729
    bs = cfg.bs if bs is None else bs
    V, blk = cfg.V, 2 * N - 1
    g = _gen(device, seed)
    f32 = torch.float32
    logits = 3.0 * torch.randn((bs, blk, V), generator=g, device=device, dtype=f32)
    p = torch.softmax(logits, -1)
    q_prev = torch.softmax(3.0 * torch.randn((bs, blk, V), generator=g, device=device,
                                             dtype=f32), -1)
    mode = (torch.rand((bs,), generator=g, device=device) < verify_frac).to(torch.int32)
    q_slot = torch.where(torch.rand((bs,), generator=g, device=device) < 0.5,
                         torch.ones((bs,), device=device, dtype=torch.int32),
                         torch.full((bs,), N, device=device, dtype=torch.int32))
    specs = torch.randint(0, V, (bs, max(N - 1, 0)), generator=g, device=device,
                          dtype=torch.int32)
    for r in range(bs):
        if int(mode[r]) != 1 or N == 1:
            continue
        qs = int(q_slot[r])
        noise = torch.randn((N - 1, V), generator=g, device=device, dtype=f32)
        rows = torch.softmax(logits[r, :N - 1] + noise, -1)
        q_prev[r, qs:qs + N - 1] = rows
        specs[r] = torch.multinomial(rows, 1, generator=g).reshape(N - 1).to(torch.int32)
    del logits
    pending = torch.randint(0, V, (bs,), generator=g, device=device, dtype=torch.int32)
    u_acc = torch.rand((bs, max(N - 1, 0)), generator=g, device=device, dtype=f32)
    u_samp = torch.rand((bs, N), generator=g, device=device, dtype=f32)
    seq_lens = torch.randint(1, 4096, (bs,), generator=g, device=device).to(torch.int32)
    return IdlmInputs(N, pending, specs.contiguous(), mode, q_slot.to(torch.int32),
                      p.contiguous(), q_prev.contiguous(), u_acc, u_samp, seq_lens)


@dataclasses.dataclass
class KvMatInputs:
    """Inputs of the draft-KV materialisation of one verify step's committed rows."""
    B: int
    n_layers: int
    Hkv: int
    D: int
    hidden: torch.Tensor        # [bs*B, H] bf16, target hidden rows
    w_kv: torch.Tensor          # [n_layers, 2, Hkv*D, H] bf16, K rows then V rows per layer
    k_norm_w: torch.Tensor      # [n_layers, D] bf16
    rope_cos: torch.Tensor      # [max_pos, D/2] fp32
    rope_sin: torch.Tensor      # [max_pos, D/2] fp32
    commit_len: torch.Tensor    # [bs] int32 in [1, B]
    seq_lens: np.ndarray        # [bs] int32, committed length before the block
    block_table: np.ndarray     # [bs, max_pages] int32
    num_pages: int
    eps: float = 1e-6


def rope_tables(max_pos: int, D: int, base: float = 1e6):
    """cos / sin tables [max_pos, D/2] of the model's rotary embedding (the
    usual frequencies base^(-2d/D), computed in fp64 and stored as fp32):
    model data handed to the call like the weights."""
    inv = base ** (-np.arange(0, D, 2, dtype=np.float64) / D)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return (torch.from_numpy(np.cos(ang).astype(np.float32)),
            torch.from_numpy(np.sin(ang).astype(np.float32)))


def make_kvmat_inputs(cfg: StepConfig, n_layers: int = 5, H: int = 4096, device="cpu",
                      seed: int | None = None, bs: int | None = None,
                      max_ctx: int | None = None) -> KvMatInputs:
    """A drafter shaped like cfg's model (Hkv, D), n_layers draft layers of
    hidden size H: hidden rows N(0, 1), projection weights N(0, 1/H) (so
    projections are about unit scale), K-norm gains 1 + 0.1 N(0, 1), all bf16;
    commit lengths uniform in [1, B]; contexts and paging as cfg's."""
    seed = (cfg.seed if seed is None else seed) + 15485863
    bs = cfg.bs if bs is None else bs
    B, Hkv, D = cfg.B, cfg.Hkv, cfg.D
    rng = np.random.default_rng(seed)
    if max_ctx is not None:
        seq_lens = rng.integers(0, max_ctx + 1, bs).astype(np.int32)
    elif bs == cfg.bs:
        seq_lens = seq_lens_for(cfg, rng)
    else:
        lo, hi = cfg.ctx[0] if isinstance(cfg.ctx[0], tuple) else (min(cfg.ctx), max(cfg.ctx))
        seq_lens = rng.integers(lo, hi + 1, bs).astype(np.int32)
    table, num_pages = paging_for(seq_lens, B, cfg.page_size, rng)
    g = _gen(device, seed)
    hidden = randn_bf16((bs * B, H), g, device)
    w = (torch.randn((n_layers, 2, Hkv * D, H), generator=g, device=device) /
         math.sqrt(H)).to(torch.bfloat16)
    kn = (1.0 + 0.1 * torch.randn((n_layers, D), generator=g, device=device)).to(torch.bfloat16)
    cos, sin = rope_tables(int(seq_lens.max()) + B + 1, D)
    commit = torch.from_numpy(rng.integers(1, B + 1, bs).astype(np.int32)).to(device)
    return KvMatInputs(B, n_layers, Hkv, D, hidden, w, kn, cos.to(device), sin.to(device),
                       commit, seq_lens, table, num_pages)


@dataclasses.dataclass
class TreeInputs:
    """A token tree per request and its verifier distributions."""
    parent: np.ndarray          # [bs, n] int32, node 0 the root (parent -1)
    block_ids: torch.Tensor     # [bs, n] int32 node tokens (root: the verified token)
    p: torch.Tensor             # [bs, n, V] fp32, verifier distribution after each node
    u: torch.Tensor             # [bs, n] fp32 uniforms by depth
    seq_lens: torch.Tensor      # [bs] int32


def random_tree_parents(rng: np.random.Generator, bs: int, n: int, window: int = 8) -> np.ndarray:
    """Bushy token trees in topological order: node i's parent is drawn from
    the `window` nodes before it, so early nodes branch and paths run deep."""
    par = np.empty((bs, n), np.int32)
    par[:, 0] = -1
    for i in range(1, n):
        lo = max(0, i - window)
        par[:, i] = rng.integers(lo, i, bs)
    return par


def psi_spec_tree_parents(rng: np.random.Generator, bs: int, n_nodes: int, block: int = 16,
                          prefixes: int = 32) -> np.ndarray:
    """Token trees shaped like the Psi-Spec Tree sampler's (B, K, V) = (16, 32,
    32): below the root (the first token, always accepted) up to `prefixes`
    drafted prefixes of block - 1 tokens, merged into a trie.  Each new prefix
    leaves an earlier one at a random depth, drawn so that exactly n_nodes
    nodes (at most 1 + prefixes * (block - 1)) result; nodes are numbered in
    creation order, which is topological."""
    depth_max = block - 1
    if not 1 <= n_nodes <= 1 + prefixes * depth_max:
        raise ValueError("n_nodes out of range for the sampler's tree")
    par = np.full((bs, n_nodes), -1, np.int32)
    for r in range(bs):
        paths: list = []
        nodes = 1
        while nodes < n_nodes:
            left = prefixes - len(paths)
            need = -(-(n_nodes - nodes) // left)  # new nodes this prefix must add at least
            if paths:
                base = paths[int(rng.integers(len(paths)))]
                s = int(rng.integers(0, min(len(base), depth_max - need) + 1))
            else:
                base, s = [], 0
            path = list(base[:s])
            prev = path[-1] if path else 0
            for _ in range(s, depth_max):
                if nodes == n_nodes:
                    break
                par[r, nodes] = prev
                path.append(nodes)
                prev = nodes
                nodes += 1
            paths.append(path)
    return par


def make_tree_inputs(cfg: StepConfig, n_nodes: int, device="cpu", seed: int | None = None,
                     bs: int | None = None, shape: str = "bushy") -> TreeInputs:
    """Trees of n_nodes nodes shaped like a top-K expansion (shape "bushy":
    random_tree_parents; "psi_spec": psi_spec_tree_parents): the children of
    a node carry the most likely tokens of its verifier distribution in rank
    order (a drafter close to the verifier).  p = softmax(2 N(0, 1) logits
    with one random token per node raised by 15), a confident verifier whose
    top token holds about three quarters of the mass at V = 151936."""
    seed = (cfg.seed if seed is None else seed) + 32452843
    bs = cfg.bs if bs is None else bs
    V = cfg.V
    rng = np.random.default_rng(seed)
    par = (psi_spec_tree_parents(rng, bs, n_nodes) if shape == "psi_spec"
           else random_tree_parents(rng, bs, n_nodes))
    g = _gen(device, seed)
    logits = 2.0 * torch.randn((bs, n_nodes, V), generator=g, device=device)
    hot = torch.randint(0, V, (bs, n_nodes, 1), generator=g, device=device)
    logits.scatter_add_(-1, hot, torch.full((bs, n_nodes, 1), 15.0, device=device))
    p = torch.softmax(logits, -1)
    del logits
    kmax = int(max(np.bincount(par[r, 1:], minlength=n_nodes).max() for r in range(bs)))
    k = min(max(kmax, 1), V)
    top = torch.topk(p, k, dim=-1).indices.cpu().numpy()  # [bs, n, k]
    ids = np.empty((bs, n_nodes), np.int32)
    ids[:, 0] = rng.integers(0, V, bs)
    for r in range(bs):
        rank = np.zeros(n_nodes, np.int64)
        for i in range(1, n_nodes):
            pa = par[r, i]
            ids[r, i] = top[r, pa, rank[pa] % k]
            rank[pa] += 1
    u = torch.rand((bs, n_nodes), generator=g, device=device)
    seq_lens = torch.randint(1, 4096, (bs,), generator=g, device=device).to(torch.int32)
    return TreeInputs(par, torch.from_numpy(ids).to(device), p.contiguous(), u, seq_lens)


def draft_from(q_rows: np.ndarray, u: np.ndarray) -> np.ndarray:
    """Inverse-CDF draws from rows of q (numpy, for small host-side workloads)."""
    c = np.cumsum(q_rows.astype(np.float64), axis=-1)
    idx = (c < (u[..., None] * c[..., -1:])).sum(-1)
    return np.minimum(idx, q_rows.shape[-1] - 1).astype(np.int32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
