#!/usr/bin/env python3
"""Benchmark one draft/verify step of block-diffusion speculative decoding.

A step is the whole hot path over one batch: prepare_block, block attention
(every pass the workload names, DRAFT and/or VERIFY) and speculative
acceptance.  Default workload: the Qwen3-8B-shaped DFlash verify step (32
requests, 32/8 heads, D 128, contexts U[1024, 4096] in 64-token pages, B = 16,
acceptance over a 151936-token vocabulary).

Prints one JSON line.  `value` is query tokens per second of whole steps with
inputs resident in HBM (device time of the step's kernels, CUDA events on the
launching stream, L2 flushed between steps); `e2e` is the same metric through
the C ABI with the step's inputs copied from pinned host memory and its result
read back every step.  `--impl reference` times the CPU oracle instead.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]
Multi-GPU (N > 1, torchrun): every rank runs an independent replica on its own
requests (the step has no cross-request exchange); the slowest rank's time
counts and value is the total over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_diffusion_speculative_attn_gb300 import workloads as wl  # noqa: E402

METRIC = "draft/verify block-attn query tokens/s + % HBM roofline; accept rows/s"
# DRAM bytes (read + write) of one attention call on the Qwen3-8B-shaped verify
# batch, from one ncu capture (summary and commands in
# profiles/qwen3_8b_verify_step_ncu.md): attention 308.42 MB read + 4.68 MB
# written (the 64-row tile merges its cut units inside the launch: no merge
# kernel).  Valid only for the kernel sources it was taken on: reported as
# null once they change.
ATTN_TRAFFIC = {"workload": "qwen3_8b_verify", "bytes_per_call": 313.04e6,
                "sources_sha256": "52d7a751db9005cea75463ba2c2cf87513cdeffcd4728d33e99fa757d08b8217"}
ATTN_SOURCES = ("block_diffusion_speculative_attn_gb300/csrc/block_attn.cu",
                "block_diffusion_speculative_attn_gb300/csrc/bdsa_device.cuh")
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
L2_CLEAN_BYTES = 256 << 20  # read after the flush: writes its dirty lines back


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="qwen3_8b_verify", choices=wl.CONFIG_ORDER)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads' attention and acceptance timings")
    ap.add_argument("--tree-only", type=int, default=0, metavar="BATCH",
                    help="time only the tree-verify attention (481-node trees) at this "
                         "batch and print its line (for profiling)")
    ap.add_argument("--only-step", action="store_true",
                    help="time the step alone: no side lines (fused append, I-DLM, KV "
                         "materialisation, tree verify), no other workloads")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# bookkeeping: algorithmic bytes / flops of one attention pass

def attn_bytes(cfg: wl.StepConfig, seq_lens: np.ndarray) -> int:
    """Each K/V element of every allowed key read once, Q read and O written once."""
    kv = int(np.sum(seq_lens.astype(np.int64) + cfg.B)) * cfg.Hkv * cfg.D * 2 * 2
    qo = 2 * cfg.bs * cfg.B * cfg.Hq * cfg.D * 2
    return kv + qo


def attn_flops(cfg: wl.StepConfig, seq_lens: np.ndarray, mode: int) -> int:
    blk = cfg.B * cfg.B if mode == wl.DRAFT else cfg.B * (cfg.B + 1) // 2
    return int(np.sum(4 * cfg.Hq * cfg.D * (cfg.B * seq_lens.astype(np.int64) + blk)))


def accept_bytes(cfg: wl.StepConfig) -> int:
    """One full row of p and q at the resolved position per request (upper bound
    of the algorithmic bytes: a fully accepted row reads p alone)."""
    return cfg.bs * 2 * cfg.V * 4 if cfg.V else 0


def accept_bytes_exact(cfg: wl.StepConfig, accept_len: np.ndarray, greedy: bool = False) -> int:
    """Algorithmic bytes of one acceptance call from its outcome.  Per row:
    the block ids, uniforms and length read and the outputs written; the (p, q)
    pairs it tests (the accepted drafts and the first rejected one); then the
    full rows the draw reads at the resolved position -- p and q for a residual
    draw after a rejection, p alone for the bonus.  Greedy reads the B rows of
    p it compares (up to the first mismatch) and the bonus row."""
    B, V = cfg.B, cfg.V
    total = 0
    for a in np.asarray(accept_len).tolist():
        total += 4 * (B + (B - 1) + 2) + 4 * (B + 4)
        if greedy:
            total += (a + 1) * V * 4
            continue
        total += 8 * min(a + 1, B - 1)
        total += (2 if a < B - 1 else 1) * V * 4
    return total


def config_dict(cfg: wl.StepConfig, world: int) -> dict:
    """The workload's description, identical on the GPU arm and the reference arm."""
    return {"workload": cfg.name, "batch": cfg.bs, "B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv,
            "D": cfg.D, "page_size": cfg.page_size,
            "ctx": list(cfg.ctx[0]) if isinstance(cfg.ctx[0], tuple) else "fixed",
            "modes": ["draft" if m == 0 else "verify" for m in cfg.modes], "vocab": cfg.V,
            "l2": "GPU arm: flushed between steps (512 MB write, then 256 MB read); "
                  "CPU reference arm: not applicable",
            "parallelism": f"replicas x{world}"}


def attn_traffic(workload: str):
    import hashlib
    h = hashlib.sha256()
    root = os.path.dirname(os.path.abspath(__file__))
    for f in ATTN_SOURCES:
        with open(os.path.join(root, f), "rb") as fh:
            h.update(fh.read())
    ok = (workload == ATTN_TRAFFIC["workload"] and
          h.hexdigest() == ATTN_TRAFFIC["sources_sha256"])
    return ATTN_TRAFFIC["bytes_per_call"] if ok else None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
class Step:
    """Device-resident inputs of one synthetic step and the calls that run it."""

    def __init__(self, cfg: wl.StepConfig, device, seed: int):
        import block_diffusion_speculative_attn_gb300 as bdsa
        self.bdsa = bdsa
        self.cfg = cfg
        self.dev = device
        self.attn = wl.make_attn_inputs(cfg, device=device, seed=seed)
        self.bt = torch.from_numpy(self.attn.block_table).to(device)
        self.sl = torch.from_numpy(self.attn.seq_lens).to(device)
        g = torch.Generator(device=device)
        g.manual_seed(seed + 17)
        V = max(cfg.V, 1)
        self.verified = torch.randint(0, V, (cfg.bs,), generator=g, device=device,
                                      dtype=torch.int32)
        self.acc = (wl.make_accept_inputs(cfg, device=device, seed=seed,
                                          seq_lens=self.attn.seq_lens) if cfg.V else None)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        B, bs = cfg.B, cfg.bs
        self.prep_out = tuple(torch.empty((bs, B), dtype=torch.int32, device=device)
                              for _ in range(3))
        self.o = torch.empty_like(self.attn.q)
        self.lse = torch.empty((bs * B, cfg.Hq), dtype=torch.float32, device=device)
        ws = bdsa.block_attn_workspace_bytes(bs, B, cfg.Hq, cfg.Hkv, cfg.D,
                                             self.attn.max_ctx_len)
        self.attn_ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=device)
        self.acc_out = None
        if cfg.V:
            self.acc_out = {k: torch.empty(bs, dtype=torch.int32, device=device)
                            for k in ("accept_len", "commit_len", "bonus_id", "new_seq_lens")}
            self.acc_out["out_tokens"] = torch.empty((bs, B), dtype=torch.int32, device=device)
            aws = bdsa.spec_accept_workspace_bytes(bs, B, cfg.V)
            self.acc_ws = torch.empty(max(aws, 256), dtype=torch.uint8, device=device)
        # kernels of ours per step: prepare, per pass the attention (cut units
        # are merged by their owner CTA inside the attention launch), accept
        self.launches = 1 + len(cfg.modes) + (1 if cfg.V else 0)

    def prepare(self):
        c = self.cfg
        self.bdsa.prepare_block(self.verified, self.sl, self.bt, self.attn.num_pages, c.B,
                                c.page_size, c.mask_token_id, out=self.prep_out,
                                dev_status=self.status)

    def attention(self, mode):
        c = self.cfg
        self.bdsa.block_attn_paged(self.attn.q, self.attn.k_cache, self.attn.v_cache, self.bt,
                                   self.sl, B=c.B, page_size=c.page_size, scale=self.attn.scale,
                                   mode=mode, max_ctx_len=self.attn.max_ctx_len,
                                   num_pages=self.attn.num_pages, out=self.o, lse=self.lse,
                                   workspace=self.attn_ws, dev_status=self.status)

    def accept(self):
        a = self.acc
        self.bdsa.spec_accept(a.block_ids, a.p, a.q, a.u_acc, a.u_samp, a.seq_lens,
                              out=self.acc_out, workspace=self.acc_ws, dev_status=self.status)

    def run(self, ev=None):
        """One step; ev = optional dict of (start, end) event pairs per stage to
        record ("attn": one pair per attention pass)."""
        self.prepare()
        for i, m in enumerate(self.cfg.modes):
            if ev is not None:
                ev["attn"][i][0].record()
            self.attention(m)
            if ev is not None:
                ev["attn"][i][1].record()
        if self.cfg.V:
            if ev is not None:
                ev["accept"][0].record()
            self.accept()
            if ev is not None:
                ev["accept"][1].record()

    # host buffers for the end-to-end measurement
    def host_inputs(self):
        pin = lambda t: t.detach().cpu().pin_memory()  # noqa: E731
        h = {"q": pin(self.attn.q), "verified": pin(self.verified), "sl": pin(self.sl),
             "bt": pin(self.bt)}
        if self.cfg.V:
            a = self.acc
            h.update({"block_ids": pin(a.block_ids), "p": pin(a.p), "qd": pin(a.q),
                      "u_acc": pin(a.u_acc), "u_samp": pin(a.u_samp)})
        return h


def run_e2e(step: Step, steps: int, warmup: int):
    """Same step, with every per-step input copied H2D from pinned memory and the
    acceptance result (or the attention output when there is no acceptance stage)
    read back D2H, all inside the timed region."""
    h = step.host_inputs()
    dev = step.dev
    d = {k: torch.empty_like(v, device=dev) for k, v in h.items()}
    res_keys = list(step.acc_out) if step.cfg.V else []
    res_host = ({k: torch.empty_like(step.acc_out[k], device="cpu").pin_memory()
                 for k in res_keys} if step.cfg.V else
                {"o": torch.empty_like(step.o, device="cpu").pin_memory()})
    h2d = sum(v.numel() * v.element_size() for v in h.values())
    d2h = sum(v.numel() * v.element_size() for v in res_host.values())
    c = step.cfg

    def one():
        for k, v in h.items():
            d[k].copy_(v, non_blocking=True)
        step.bdsa.prepare_block(d["verified"], d["sl"], d["bt"], step.attn.num_pages, c.B,
                                c.page_size, c.mask_token_id, out=step.prep_out)
        for m in c.modes:
            step.bdsa.block_attn_paged(d["q"], step.attn.k_cache, step.attn.v_cache, d["bt"],
                                       d["sl"], B=c.B, page_size=c.page_size,
                                       scale=step.attn.scale, mode=m,
                                       max_ctx_len=step.attn.max_ctx_len,
                                       num_pages=step.attn.num_pages, out=step.o,
                                       workspace=step.attn_ws)
        if c.V:
            step.bdsa.spec_accept(d["block_ids"], d["p"], d["qd"], d["u_acc"], d["u_samp"],
                                  d["sl"], out=step.acc_out, workspace=step.acc_ws)
            for k in res_keys:
                res_host[k].copy_(step.acc_out[k], non_blocking=True)
        else:
            res_host["o"].copy_(step.o, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return ms, h2d, d2h


def time_fused_append(step: Step, flush, clean, iters: int = 20):
    """The attention call with and without the fused block-KV append (the
    block's own keys and values written into the paged cache by the same
    launch), interleaved, L2 flushed before each; mean event times in ms."""
    c = step.cfg
    g = torch.Generator(device=step.dev)
    g.manual_seed(c.seed + 99)
    shape = (c.bs * c.B, c.Hkv, c.D)
    k_new = torch.randn(shape, generator=g, device=step.dev).to(torch.bfloat16)
    v_new = torch.randn(shape, generator=g, device=step.dev).to(torch.bfloat16)
    mode = c.modes[-1]

    def call(append):
        step.bdsa.block_attn_paged(step.attn.q, step.attn.k_cache, step.attn.v_cache, step.bt,
                                   step.sl, B=c.B, page_size=c.page_size, scale=step.attn.scale,
                                   mode=mode, max_ctx_len=step.attn.max_ctx_len,
                                   num_pages=step.attn.num_pages, out=step.o, lse=step.lse,
                                   workspace=step.attn_ws, dev_status=step.status,
                                   k_new=k_new if append else None,
                                   v_new=v_new if append else None)

    times = {False: [], True: []}
    for i in range(iters + 2):
        for append in ((False, True) if i % 2 == 0 else (True, False)):
            flush.zero_()
            clean.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call(append)
            e1.record()
            if i >= 2:
                times[append].append((e0, e1))
    torch.cuda.synchronize()
    ms = {a: statistics.mean(x.elapsed_time(y) for x, y in v) for a, v in times.items()}
    return {"launch_ms": ms[True], "plain_launch_ms": ms[False],
            "added_us": (ms[True] - ms[False]) * 1e3,
            "bytes_written": 2 * c.bs * c.B * c.Hkv * c.D * 2, "iters": iters}


def idlm_bytes(mode: np.ndarray, accept_len: np.ndarray, N: int, V: int) -> int:
    """Algorithmic bytes of one I-DLM round's acceptance: per request, the
    gathered p / q pairs of the tested specs, then every distribution row a
    draw reads: p and q_prev at a rejection (the residual), p alone for a bonus
    or a cold start's clean token, and one p row per new spec drawn."""
    total = 0
    for m, a in zip(mode.tolist(), accept_len.tolist()):
        if m == 1:
            total += 2 * 4 * (a + 1 if a < N - 1 else N - 1)
            rows = 2 if a < N - 1 else N
        else:
            rows = N
        total += rows * V * 4
    return total


def time_idlm(cfg: wl.StepConfig, dev, flush, clean, N: int = 8, iters: int = 20,
              cpu: bool = False):
    """The I-DLM Block-N round at the workload's batch and vocabulary: layout
    (idlm_prepare) and verify / correct / new-spec draws (idlm_accept), L2
    flushed before each round; mean event times in ms."""
    import block_diffusion_speculative_attn_gb300 as bdsa
    x = wl.make_idlm_inputs(cfg, N=N, device=dev)
    blk = 2 * N - 1
    rng = np.random.default_rng(cfg.seed + 5)
    table, num_pages = wl.paging_for(x.seq_lens.cpu().numpy(), blk, cfg.page_size, rng)
    bt = torch.from_numpy(table).to(dev)
    bs = cfg.bs
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    prep = tuple(torch.empty((bs, blk), dtype=torch.int32, device=dev) for _ in range(3))
    out = {k: torch.empty(bs, dtype=torch.int32, device=dev) for k in bdsa.IDLM_KEYS}
    out["out_tokens"] = torch.empty((bs, N), dtype=torch.int32, device=dev)
    out["next_specs"] = torch.empty((bs, N - 1), dtype=torch.int32, device=dev)
    times = []
    for i in range(iters + 3):
        flush.zero_()
        clean.sum()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record()
        bdsa.idlm_prepare(x.pending, x.specs, x.mode, x.seq_lens, bt, num_pages, N,
                          cfg.page_size, cfg.mask_token_id, out=prep, dev_status=status)
        ev[1].record()
        bdsa.idlm_accept(prep[0], x.mode, x.p, x.q_prev, x.q_slot, x.u_acc, x.u_samp,
                         x.seq_lens, N, out=out, dev_status=status)
        ev[2].record()
        if i >= 3:
            times.append(ev)
    torch.cuda.synchronize()
    assert status.item() == 0, bdsa.STATUS.get(status.item())
    round_ms = statistics.mean(e[0].elapsed_time(e[2]) for e in times)
    acc_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in times)
    mode = x.mode.cpu().numpy()
    a = out["accept_len"].cpu().numpy()
    nbytes = idlm_bytes(mode, a, N, cfg.V)
    hbm, _, src = peaks()
    achieved = nbytes / (acc_ms / 1e3) / 1e9
    base = None
    if cpu:
        # the oracle on every row of the same round, on the host cores
        import oracle
        cores = len(os.sched_getaffinity(0))
        host = [t.cpu().numpy() for t in (prep[0], x.mode, x.p, x.q_prev, x.q_slot, x.u_acc,
                                          x.u_samp, x.seq_lens)]
        t0 = time.perf_counter()
        oracle.idlm_accept(*host, N, nthreads=cores)
        dt = time.perf_counter() - t0
        base = {"value": bs / dt, "unit": "rows/s", "cores": cores, "kind": "oracle",
                "sample": f"all {bs} rows of the round, fp64/fp32 C oracle, {cores} threads",
                "seconds": dt}
    return {"N": N, "slots": blk, "batch": bs, "vocab": cfg.V,
            "verify_share": float(mode.mean()), "mean_accept_len": float(a[mode == 1].mean()),
            "cpu_baseline": base,
            "round_ms": round_ms, "accept_ms": acc_ms, "rows_per_s": bs / (acc_ms / 1e3),
            "accept_roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm,
                                "unit": "GB/s", "frac": achieved / hbm, "peak_source": src,
                                "algorithmic_bytes_per_launch": nbytes},
            "gpu_launches_per_round": 2, "iters": iters}


def kvmat_bytes(rows: int, H: int, n_layers: int, Hkv: int, D: int) -> int:
    """Algorithmic bytes of one KV materialisation: every projection weight
    read once, each committed hidden row read once, its K and V written once."""
    return (n_layers * 2 * Hkv * D * H * 2 + rows * H * 2 + rows * n_layers * 2 * Hkv * D * 2)


def time_kvmat(step: "Step", flush, clean, n_layers: int = 5, H: int = 4096, iters: int = 20,
               cpu: bool = False):
    """The draft KV materialisation of this step's committed rows (commit_len
    from the step's acceptance, positions and slots from its prepare_block)
    for a drafter of n_layers layers of hidden size H with the model's KV
    heads, into a draft pool paged like the target cache; L2 flushed before
    each call; mean event time in ms."""
    import block_diffusion_speculative_attn_gb300 as bdsa
    c = step.cfg
    x = wl.make_kvmat_inputs(c, n_layers=n_layers, H=H, device=step.dev)
    slots = step.attn.num_pages * c.page_size
    kc = torch.empty((n_layers, slots, c.Hkv, c.D), dtype=torch.bfloat16, device=step.dev)
    vc = torch.empty_like(kc)
    ws = torch.empty(bdsa.kv_materialize_workspace_bytes(c.bs, c.B, H), dtype=torch.uint8,
                     device=step.dev)
    commit = step.acc_out["commit_len"]
    pos = step.prep_out[1].reshape(-1)
    loc = step.prep_out[2].reshape(-1)
    status = torch.zeros(1, dtype=torch.int32, device=step.dev)
    times = []
    for i in range(iters + 3):
        flush.zero_()
        clean.sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        bdsa.kv_materialize(x.hidden, commit, pos, loc, x.w_kv, x.k_norm_w, x.rope_cos,
                            x.rope_sin, kc, vc, B=c.B, eps=x.eps, workspace=ws,
                            dev_status=status)
        e1.record()
        if i >= 3:
            times.append((e0, e1))
    torch.cuda.synchronize()
    assert status.item() == 0, bdsa.STATUS.get(status.item())
    ms = statistics.mean(a.elapsed_time(b) for a, b in times)
    rows = int(commit.sum().item())
    nbytes = kvmat_bytes(rows, H, n_layers, c.Hkv, c.D)
    flops = 2 * rows * H * n_layers * 2 * c.Hkv * c.D
    hbm, tf, src = peaks()
    achieved = nbytes / (ms / 1e3) / 1e9
    base = None
    if cpu:
        # the oracle on the committed rows of the first requests (about 2 s)
        import oracle
        cores = len(os.sched_getaffinity(0))
        cl = commit.cpu().numpy()
        hb, wb, gb = wl.bf16_bits(x.hidden), wl.bf16_bits(x.w_kv), wl.bf16_bits(x.k_norm_w)
        args = (pos.cpu().numpy(), loc.cpu().numpy())
        keep = np.zeros_like(cl)
        n, dt = 0, 0.0
        while n < c.bs and dt < 0.5:
            n = min(c.bs, max(1, 2 * n))
            keep[:] = 0
            keep[:n] = cl[:n]
            t0 = time.perf_counter()
            oracle.kv_materialize(hb, keep, *args, wb, gb, x.rope_cos.cpu().numpy(),
                                  x.rope_sin.cpu().numpy(), x.eps, c.B, n_layers, c.Hkv, c.D,
                                  slots, nthreads=cores)
            dt = time.perf_counter() - t0
        base = {"value": int(keep.sum()) / dt, "unit": "rows/s", "cores": cores,
                "kind": "oracle",
                "sample": f"the committed rows of the first {n} of {c.bs} requests "
                          f"({int(keep.sum())} rows), fp64 C oracle, {cores} threads",
                "seconds": dt}
    return {"n_layers": n_layers, "hidden": H, "committed_rows": rows, "launch_ms": ms,
            "cpu_baseline": base,
            "rows_per_s": rows / (ms / 1e3), "tflops": flops / (ms / 1e3) / 1e12,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_source": src,
                         "algorithmic_bytes_per_launch": nbytes, "flops_per_launch": flops},
            "gpu_launches_per_call": 2, "iters": iters}


def tree_attn_flops(c: wl.StepConfig, seq_lens: np.ndarray, depth: np.ndarray) -> int:
    """Algorithmic FLOPs of tree attention: every query row (request r, node i,
    query head) against the L_r + depth(i) + 1 keys it sees, QK^T and PV at
    2 FLOPs a multiply-add each."""
    keys = seq_lens.astype(np.int64)[:, None] + depth.astype(np.int64) + 1
    return int(keys.sum()) * c.Hq * c.D * 4


def time_tree(cfg: wl.StepConfig, dev, flush, clean, n_nodes: int = 481, iters: int = 10,
              cpu: bool = False, accept: bool = True):
    """Tree verify at the workload's shape with token trees shaped like the
    Psi-Spec Tree sampler's (B, K, V) = (16, 32, 32): 32 prefixes of 15 drafted
    tokens under the root, n_nodes = 481 nodes.  Times the layout
    (tree_prepare) plus tree attention over the paged cache (row tiles of
    128 / G nodes), and the tree acceptance walk over the vocabulary; L2
    flushed before each call; mean event times in ms.  The attention is bound
    by the tensor cores at this size (each key serves G * 481 query rows)."""
    import dataclasses

    import block_diffusion_speculative_attn_gb300 as bdsa
    c = dataclasses.replace(cfg, B=n_nodes)
    attn = wl.make_attn_inputs(c, device=dev, seed=c.seed + 77)
    bt = torch.from_numpy(attn.block_table).to(dev)
    sl = torch.from_numpy(attn.seq_lens).to(dev)
    if accept:
        x = wl.make_tree_inputs(cfg, n_nodes, device=dev, shape="psi_spec")
        parents = x.parent
    else:
        parents = wl.psi_spec_tree_parents(np.random.default_rng(c.seed + 32452843), c.bs,
                                           n_nodes)
    par = torch.from_numpy(parents).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    prep = tuple(torch.empty((c.bs, n_nodes), dtype=torch.int32, device=dev) for _ in range(3)) \
        + (torch.empty((c.bs, n_nodes, bdsa.tree_mask_words(n_nodes)), dtype=torch.int64,
                       device=dev),)
    out = torch.empty_like(attn.q)
    ws = torch.empty(max(bdsa.block_attn_workspace_bytes(c.bs, c.B, c.Hq, c.Hkv, c.D,
                                                         attn.max_ctx_len), 256),
                     dtype=torch.uint8, device=dev)
    acc = {k: torch.empty(c.bs, dtype=torch.int32, device=dev) for k in bdsa.TREE_KEYS}
    acc["path"] = torch.empty((c.bs, n_nodes), dtype=torch.int32, device=dev)
    acc["out_tokens"] = torch.empty((c.bs, n_nodes), dtype=torch.int32, device=dev)
    t_attn, t_acc = [], []
    for i in range(iters + 3):
        flush.zero_()
        clean.sum()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record()
        bdsa.tree_prepare(par, sl, bt, attn.num_pages, c.page_size, out=prep, dev_status=status)
        bdsa.block_attn_paged(attn.q, attn.k_cache, attn.v_cache, bt, sl, B=c.B,
                              page_size=c.page_size, scale=attn.scale, mode=wl.VERIFY,
                              max_ctx_len=attn.max_ctx_len, num_pages=attn.num_pages, out=out,
                              workspace=ws, dev_status=status, tree_mask=prep[3])
        ev[1].record()
        flush.zero_()
        clean.sum()
        ev2 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev2[0].record()
        if accept:
            bdsa.tree_accept(x.block_ids, par, x.p, x.u, x.seq_lens, out=acc, dev_status=status)
        ev2[1].record()
        if i >= 3:
            t_attn.append(ev[:2])
            t_acc.append(ev2)
    torch.cuda.synchronize()
    assert status.item() == 0, bdsa.STATUS.get(status.item())
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in t_attn)
    acc_ms = statistics.mean(a.elapsed_time(b) for a, b in t_acc)
    hbm, tf, src = peaks()
    abytes = attn_bytes(c, attn.seq_lens)
    aflops = tree_attn_flops(c, attn.seq_lens, prep[0].cpu().numpy())
    depth = acc["accept_len"].cpu().numpy() if accept else np.zeros(c.bs, np.int64)
    accbytes = int((depth + 1).sum()) * cfg.V * 4
    base = None
    if cpu and accept:
        # the oracle: tree attention of the first request, acceptance of the
        # first four rows
        import oracle
        cores = len(os.sched_getaffinity(0))
        ps = c.page_size
        need = (int(attn.seq_lens[0]) + c.B + ps - 1) // ps
        idx = torch.from_numpy(attn.block_table[0, :need].astype(np.int64)).to(dev)
        kc = attn.k_cache.view(-1, ps, c.Hkv, c.D)[idx].reshape(-1, c.Hkv, c.D)
        vc = attn.v_cache.view(-1, ps, c.Hkv, c.D)[idx].reshape(-1, c.Hkv, c.D)
        qb = wl.bf16_bits(attn.q[:c.B])
        kb, vb = wl.bf16_bits(kc), wl.bf16_bits(vc)
        t0 = time.perf_counter()
        oracle.block_attn_tree(qb, kb, vb, np.arange(need, dtype=np.int32)[None],
                               attn.seq_lens[:1], x.parent[:1], c.B, c.Hq, c.Hkv, c.D, ps,
                               attn.scale, num_pages=need, nthreads=cores)
        dt_attn = time.perf_counter() - t0
        na = min(4, c.bs)
        host = [x.block_ids[:na].cpu().numpy(), x.parent[:na], x.p[:na].cpu().numpy(),
                x.u[:na].cpu().numpy(), x.seq_lens[:na].cpu().numpy()]
        t0 = time.perf_counter()
        oracle.tree_accept(*host, nthreads=cores)
        dt_acc = time.perf_counter() - t0
        base = {"value": n_nodes / dt_attn, "unit": "query tokens/s (tree attention)",
                "accept_rows_per_s": na / dt_acc, "cores": cores, "kind": "oracle",
                "sample": f"tree attention of 1 of {c.bs} requests, acceptance of {na} "
                          f"rows, fp64 C oracle, {cores} threads",
                "seconds": dt_attn + dt_acc}
    tach = aflops / (attn_ms / 1e3) / 1e12
    if not accept:
        acc_ms = None
    return {"nodes": n_nodes, "tree": "Psi-Spec (16, 32, 32): 32 prefixes of 15 tokens",
            "batch": c.bs, "vocab": cfg.V, "cpu_baseline": base,
            "attn_ms": attn_ms, "attn_query_tokens_per_s": c.bs * n_nodes / (attn_ms / 1e3),
            "attn_roofline": {"bound": "tensor", "achieved": tach, "peak": tf,
                              "unit": "TFLOP/s", "frac": tach / tf, "peak_source": src,
                              "algorithmic_flops_per_launch": aflops,
                              "hbm_achieved_gbs": abytes / (attn_ms / 1e3) / 1e9,
                              "algorithmic_bytes_per_launch": abytes,
                              "kernels": "tree_prepare + block attention (TREE) + merge"},
            "accept_ms": acc_ms,
            "accept_rows_per_s": c.bs / (acc_ms / 1e3) if acc_ms else None,
            "mean_accept_len": float(depth.mean()) if accept else None,
            "accept_roofline": None if not accept else {
                "bound": "hbm", "achieved": accbytes / (acc_ms / 1e3) / 1e9, "peak": hbm,
                "unit": "GB/s", "frac": accbytes / (acc_ms / 1e3) / 1e9 / hbm,
                "peak_source": src, "algorithmic_bytes_per_launch": accbytes},
            "iters": iters}


OTHER_WORKLOADS = ("llada2_block_draft", "uno_1k8k_step", "long_ctx_verify")


def time_workload(name: str, dev, flush, clean, iters: int = 10, cpu: bool = False):
    """Another workload's step: every attention pass (DRAFT and / or VERIFY)
    and the acceptance, each timed alone with CUDA events (L2 flushed before
    every step), with its algorithmic bytes against the HBM peak; the step
    itself is timed again without events between its kernels."""
    cfg = wl.config(name)
    st = Step(cfg, dev, seed=cfg.seed)
    hbm, _, src = peaks()
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))  # noqa: E731
    for _ in range(3):
        flush.zero_()
        clean.sum()
        st.run()
    torch.cuda.synchronize()
    assert st.status.item() == 0, st.bdsa.STATUS.get(st.status.item())
    step_ev = []
    for _ in range(iters):
        flush.zero_()
        clean.sum()
        e = mk()
        e[0].record()
        st.run()
        e[1].record()
        step_ev.append(e)
    stage_ev = []
    for _ in range(iters):
        flush.zero_()
        clean.sum()
        ev = {"attn": [mk() for _ in cfg.modes], "accept": mk()}
        st.run(ev)
        stage_ev.append(ev)
    torch.cuda.synchronize()
    step_ms = statistics.mean(a.elapsed_time(b) for a, b in step_ev)
    abytes = attn_bytes(cfg, st.attn.seq_lens)
    passes = []
    for j, m in enumerate(cfg.modes):
        ms = statistics.mean(e["attn"][j][0].elapsed_time(e["attn"][j][1]) for e in stage_ev)
        ach = abytes / (ms / 1e3) / 1e9
        passes.append({"mode": "draft" if m == wl.DRAFT else "verify", "launch_ms": ms,
                       "query_tokens_per_s": cfg.bs * cfg.B / (ms / 1e3),
                       "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                                    "frac": ach / hbm, "peak_source": src,
                                    "algorithmic_bytes_per_launch": abytes,
                                    "flops_per_launch": attn_flops(cfg, st.attn.seq_lens, m)}})
    acc = None
    if cfg.V:
        ms = statistics.mean(e["accept"][0].elapsed_time(e["accept"][1]) for e in stage_ev)
        nb = accept_bytes_exact(cfg, st.acc_out["accept_len"].cpu().numpy())
        ach = nb / (ms / 1e3) / 1e9
        acc = {"launch_ms": ms, "rows_per_s": cfg.bs / (ms / 1e3),
               "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                            "frac": ach / hbm, "peak_source": src,
                            "algorithmic_bytes_per_launch": nb}}
    base = None
    if cpu:
        # the oracle's whole step on the first request, best of 3
        cores = len(os.sched_getaffinity(0))
        smp = oracle_sample(cfg, st.attn, st.acc, [0], cores)
        times = []
        for _ in range(3):
            t0 = time.perf_counter()
            oracle_step(cfg, smp, st.attn.scale, cores)
            times.append(time.perf_counter() - t0)
        best = min(times)
        base = {"value": cfg.B * len(cfg.modes) / best, "unit": "query tokens/s",
                "cores": cores, "kind": "oracle",
                "sample": f"first 1 of {cfg.bs} requests of {cfg.name}, whole step, fp64 C "
                          f"oracle, {cores} OpenMP threads, best of 3", "seconds": best}
    out = {"config": config_dict(cfg, 1), "step_ms": step_ms,
           "query_tokens_per_s": cfg.bs * cfg.B * len(cfg.modes) / (step_ms / 1e3),
           "attention_passes": passes, "accept": acc, "cpu_baseline": base, "iters": iters,
           "gpu_launches_per_step": st.launches}
    del st
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
def oracle_sample(cfg: wl.StepConfig, attn: wl.AttnInputs, acc, reqs, nthreads):
    """Host copies of the sampled requests' inputs (compact page pool)."""
    ps = cfg.page_size
    need = [(int(attn.seq_lens[r]) + cfg.B + ps - 1) // ps for r in reqs]
    pages = np.concatenate([attn.block_table[r, :n] for r, n in zip(reqs, need)])
    idx = torch.from_numpy(pages.astype(np.int64)).to(attn.k_cache.device)
    kc = attn.k_cache.view(-1, ps, cfg.Hkv, cfg.D)[idx].reshape(-1, cfg.Hkv, cfg.D)
    vc = attn.v_cache.view(-1, ps, cfg.Hkv, cfg.D)[idx].reshape(-1, cfg.Hkv, cfg.D)
    table = np.full((len(reqs), max(need)), -1, np.int32)
    at = 0
    for j, n in enumerate(need):
        table[j, :n] = np.arange(at, at + n, dtype=np.int32)
        at += n
    rows = torch.cat([torch.arange(r * cfg.B, (r + 1) * cfg.B) for r in reqs]).to(attn.q.device)
    s = {"q": wl.bf16_bits(attn.q[rows]), "k": wl.bf16_bits(kc), "v": wl.bf16_bits(vc),
         "table": table, "num_pages": at, "seq_lens": attn.seq_lens[reqs].copy(),
         "verified": np.zeros(len(reqs), np.int32)}
    if acc is not None:
        rt = torch.as_tensor(reqs, device=acc.p.device)
        s.update({"block_ids": acc.block_ids[rt].cpu().numpy(), "p": acc.p[rt].cpu().numpy(),
                  "qd": acc.q[rt].cpu().numpy(), "u_acc": acc.u_acc[rt].cpu().numpy(),
                  "u_samp": acc.u_samp[rt].cpu().numpy(),
                  "acc_sl": acc.seq_lens[rt].cpu().numpy()})
    return s


def oracle_step(cfg: wl.StepConfig, s, scale, nthreads):
    import oracle
    oracle.prepare_block(s["verified"], s["seq_lens"], s["table"], s["num_pages"], cfg.B,
                         cfg.page_size, cfg.mask_token_id)
    for m in cfg.modes:
        oracle.block_attn(s["q"], s["k"], s["v"], s["table"], s["seq_lens"], cfg.B, cfg.Hq,
                          cfg.Hkv, cfg.D, cfg.page_size, scale, m, num_pages=s["num_pages"],
                          nthreads=nthreads)
    if cfg.V:
        oracle.spec_accept(s["block_ids"], s["p"], s["qd"], s["u_acc"], s["u_samp"], s["acc_sl"],
                           nthreads=nthreads)


def cpu_baseline(cfg, attn, acc, target_s: float, reps: int = 3):
    """Time the oracle on a bounded sample of the same workload on the host cores."""
    cores = len(os.sched_getaffinity(0))
    # grow the sample of requests until one oracle step takes a measurable time
    n = 1
    while True:
        reqs = list(range(min(n, cfg.bs)))
        s = oracle_sample(cfg, attn, acc, reqs, cores)
        t0 = time.perf_counter()
        oracle_step(cfg, s, attn.scale, cores)
        dt = time.perf_counter() - t0
        if dt * 4 > target_s or n >= cfg.bs:
            break
        n = min(cfg.bs, max(n + 1, int(n * max(2.0, 0.5 * target_s / max(dt, 1e-3)))))
    times = [dt]
    for _ in range(reps - 1):
        t0 = time.perf_counter()
        oracle_step(cfg, s, attn.scale, cores)
        times.append(time.perf_counter() - t0)
    best = min(times)
    tokens = len(reqs) * cfg.B * len(cfg.modes)
    return {"value": tokens / best, "unit": "query tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {len(reqs)} of {cfg.bs} requests of {cfg.name}, whole step "
                      f"(prepare, {len(cfg.modes)} attention pass(es)"
                      f"{', acceptance' if cfg.V else ''}), fp64 C oracle, "
                      f"{cores} OpenMP threads, best of {len(times)}",
            "seconds": best, "requests": len(reqs)}


# ---------------------------------------------------------------------------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main_reference(args, world, rank):
    """Reference arm: the CPU oracle as it stands, on bounded samples of the workload."""
    if rank != 0:
        return
    cfg = wl.config(args.workload)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    attn = wl.make_attn_inputs(cfg, device=dev, seed=cfg.seed)
    acc = wl.make_accept_inputs(cfg, device=dev, seed=cfg.seed,
                                seq_lens=attn.seq_lens) if cfg.V else None
    cores = len(os.sched_getaffinity(0))
    # sample size: requests whose oracle step takes ~ cpu_seconds / (steps + warmup)
    per_step = max(0.5, args.cpu_seconds * 8 / max(1, args.steps + args.warmup))
    probe = cpu_baseline(cfg, attn, acc, per_step)
    reqs = list(range(probe["requests"]))
    s = oracle_sample(cfg, attn, acc, reqs, cores)
    for _ in range(args.warmup):
        oracle_step(cfg, s, attn.scale, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(cfg, s, attn.scale, cores)
    dt = (time.perf_counter() - t0) / args.steps
    tokens = len(reqs) * cfg.B * len(cfg.modes)
    value = tokens / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "query tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(cfg, world),
            "cpu_baseline": {"value": value, "unit": "query tokens/s", "cores": cores,
                             "kind": "oracle",
                             "sample": f"first {len(reqs)} of {cfg.bs} requests per step",
                             "requests_per_step": len(reqs)},
            "e2e": {"value": value, "unit": "query tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        main_reference(args, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import block_diffusion_speculative_attn_gb300 as bdsa
    bdsa.lib()
    cfg = wl.config(args.workload)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32, device=dev)
    if args.tree_only:
        import dataclasses
        tc = dataclasses.replace(cfg, bs=args.tree_only)
        print(json.dumps({"tree_verify": time_tree(tc, dev, flush, clean, iters=args.steps,
                                                   accept=False)}), flush=True)
        return
    step = Step(cfg, dev, seed=cfg.seed + 1000 * rank)
    K = args.steps
    ev = [{"step": (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)),
           "attn": [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in cfg.modes],
           "accept": (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))}
          for _ in range(K)]
    # The clock sampler starts first; the warm-up steps then run right before
    # the timed ones, so the GPU does not sit idle in between (an idle gap made
    # the first timed step an outlier).
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        clean.sum()
        step.run()
    torch.cuda.synchronize()
    assert step.status.item() == 0, bdsa.STATUS.get(step.status.item())
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        # Evict the previous step's lines from L2 (outside the events): write a
        # buffer larger than L2, then read another one so that the write-back
        # of the flush's own dirty lines does not land inside the next step.
        flush.zero_()
        clean.sum()
        ev[i]["step"][0].record()
        step.run()
        ev[i]["step"][1].record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    # The stages' own times come from a second pass of K steps with events
    # between the stages (an event between two kernels keeps the second from
    # starting while the first finishes, so the step time above has none).
    for i in range(K):
        flush.zero_()
        clean.sum()
        step.run(ev[i])
    torch.cuda.synchronize()
    step_ms = [e["step"][0].elapsed_time(e["step"][1]) for e in ev]
    ms = statistics.mean(step_ms)
    # mean time of one attention call (over the steps and the step's passes)
    attn_ms = statistics.mean(a.elapsed_time(b) for e in ev for a, b in e["attn"])
    acc_ms = (statistics.mean(e["accept"][0].elapsed_time(e["accept"][1]) for e in ev)
              if cfg.V else None)
    ms_max = max_over_ranks(ms, world, dev)

    tokens = cfg.bs * cfg.B * len(cfg.modes)
    value = tokens * world / (ms_max / 1e3)
    hbm, tf, peak_src = peaks()
    abytes = attn_bytes(cfg, step.attn.seq_lens)
    roof = None
    if attn_ms is not None:
        achieved = abytes / (attn_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": attn_traffic(cfg.name),
                "kernel": "block_attn_paged (one launch: the owner CTA of each cut unit "
                          "merges it)",
                "algorithmic_bytes_per_launch": abytes, "peak_source": peak_src,
                "launch_ms": attn_ms}

    acc_roof = None
    if acc_ms:
        nb = accept_bytes_exact(cfg, step.acc_out["accept_len"].cpu().numpy())
        ach = nb / (acc_ms / 1e3) / 1e9
        acc_roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                    "frac": ach / hbm, "peak_source": peak_src,
                    "kernel": "spec_accept (stochastic)", "algorithmic_bytes_per_launch": nb,
                    "launch_ms": acc_ms}

    # the side lines run on single-pass workloads (the default one included)
    single = len(cfg.modes) == 1
    fused_append = None
    if single and not args.only_step:
        fused_append = time_fused_append(step, flush, clean)
        assert step.status.item() == 0, bdsa.STATUS.get(step.status.item())
    side = cfg.V and single and not args.only_step
    cpu_side = rank == 0 and world == 1 and not args.no_cpu_baseline
    idlm = time_idlm(cfg, dev, flush, clean, cpu=cpu_side) if side else None
    kvmat = time_kvmat(step, flush, clean, cpu=cpu_side) if side else None
    tree = time_tree(cfg, dev, flush, clean, cpu=cpu_side) if side else None
    # the other workloads' attention passes (draft mode among them) and acceptance
    others = None
    if cfg.name == "qwen3_8b_verify" and not (args.no_workloads or args.only_step):
        others = {n: time_workload(n, dev, flush, clean, cpu=cpu_side) for n in OTHER_WORKLOADS}

    e2e = None
    if not args.no_e2e:
        e_ms, h2d, d2h = run_e2e(step, max(3, K // 2), 2)
        e_ms = max_over_ranks(e_ms, world, dev)
        e2e = {"value": tokens * world / (e_ms / 1e3), "unit": "query tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, step.attn, step.acc, args.cpu_seconds)

    line = {"metric": METRIC, "value": value, "unit": "query tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_dict(cfg, world),
            "roofline": roof,
            "attn_query_tokens_per_s": (cfg.bs * cfg.B / (attn_ms / 1e3)) if attn_ms else None,
            "accept_rows_per_s": (cfg.bs / (acc_ms / 1e3)) if acc_ms else None,
            "accept_ms": acc_ms,
            "accept_roofline": acc_roof,
            "workloads": others,
            "fused_append": fused_append,
            "idlm_round": idlm,
            "kv_materialize": kvmat,
            "tree_verify": tree,
            "attn_flops_per_launch": attn_flops(cfg, step.attn.seq_lens, cfg.modes[-1]),
            "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": step.launches * K,
            "clocks": clk}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
