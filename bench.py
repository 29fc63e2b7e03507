"""Benchmark: the fused decoder-op chain of one Qwen-7B-like layer, fwd+bwd.

One step runs every operator once, forward and backward, on independently
drawn bf16 tensors of the layer's shapes at batch 1, seq S (default 32768):

  RMSNorm fwd [S, 4096] -> RoPE fwd Q/K [1, S, 32, 128] -> SwiGLU fwd [S, 11008]
  -> fused linear-CE fwd+bwd (S x 4096 x 151936, 10 % ignored labels)
  -> SwiGLU bwd -> RoPE bwd -> RMSNorm bwd

Prints one JSON line: tokens/s of the whole chain (device-resident inputs),
the same through host buffers (e2e), the roofline of the dominant kernel
(the linear-CE's tensor-core GEMMs, 6*S*H*V algorithmic flops per call),
HBM GB/s of every memory-bound kernel, the oracle's CPU throughput on a
bounded sample, and SM clocks sampled during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--seq S] [--impl reference]

Beside the headline chain, the line carries one entry per named workload
("configs"): per-operator latency of the tiny set (fp32 and bf16), HBM GB/s of
SwiGLU at [4, 2048, 11008] and of RMSNorm / RoPE at the Llama-3-8B shapes,
tokens/s and tensor-core fraction of the fused linear-CE at the Llama-3 head
(8192 x 4096 x 128256), and the chain's tokens/s at seq 512 / 2048 / 8192.

Under torchrun (N > 1) every rank runs its own chain on its own data (weak
scaling, no collective on the data path); the timed region is bracketed by
barriers and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HIDDEN, HEADS, HEAD_DIM, INTER, VOCAB = 4096, 32, 128, 11008, 151936
THETA, EPS = 1e4, 1e-6
PARAMETERS = ("w", "W")   # RMSNorm weight, lm_head weight: resident across steps
METRIC = "fused decoder-op chain tokens/s fwd+bwd (RMSNorm, RoPE, SwiGLU, fused linear-CE)"
UNIT = "tokens/s"


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--seq", type=int, default=32768)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-configs", action="store_true", help="skip the per-workload entries (configs)")
    p.add_argument("--op", default="chain",
                   choices=["chain", "linear_ce", "linear_ce_two_pass", "rmsnorm_qkv_rope", "fused_linear_swiglu",
                            "fused_linear_swiglu_fwd_save", "fused_linear_swiglu_bwd_saved", "rmsnorm", "rope",
                            "swiglu"],
                   help="chain: the benchmark step (default); otherwise time that one operator alone at --seq "
                        "tokens (single-kernel profiling cases; prints a JSON line with ms per call)")
    p.add_argument("--chunk", type=int, default=0, help="--op linear_ce: token chunk (0 = automatic)")
    p.add_argument("--ignore-frac", type=float, default=0.1,
                   help="--op linear_ce / linear_ce_two_pass: fraction of labels set to ignore_index")
    return p.parse_args(argv)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


# ------------------------------------------------------------------ ranks
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """Slowest rank's time (the job's time); identity on one process."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, dist, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


class DataParallel:
    """The exchanges of a token-sharded (data-parallel) step, over one process
    per GPU: every rank holds its own tokens, the operators run on them with no
    exchange, and only what the mean and the weight gradients imply crosses
    ranks -- the count of non-ignored labels (all ranks' sum) before the fused
    linear-CE, which then runs in sum mode with grad_scale = 1 / that count,
    and after the backward the sums of the loss, of dW [V, H] and of the
    RMSNorm dw [H].  dX, dx and the other operators' gradients stay local.
    n_local is this rank's count of non-ignored labels (known on the host,
    where the labels come from)."""

    def __init__(self, dist, n_local, device):
        self.dist, self.n_local, self.device = dist, int(n_local), device
        self.n_global = None

    def valid_count(self) -> int:
        import torch
        t = torch.tensor([self.n_local], dtype=torch.int64, device=self.device)
        self.dist.all_reduce(t)
        self.n_global = int(t.item())
        return self.n_global

    def reduce_grads(self, loss, dW, dw):
        for t in (loss, dW, dw):
            self.dist.all_reduce(t)

    def mean_loss(self, loss_sum: float) -> float:
        return loss_sum / self.n_global if self.n_global else 0.0


# ---------------------------------------------------------------- workload
def workload_config(S):
    return {"workload": f"Qwen-7B-like layer op chain, batch 1, seq {S}: RMSNorm [{S}x{HIDDEN}] -> RoPE Q/K "
                        f"[1,{S},{HEADS},{HEAD_DIM}] -> SwiGLU [{S}x{INTER}] -> fused linear-CE "
                        f"{S}x{HIDDEN}x{VOCAB}, fwd+bwd",
            "batch": 1, "seq_len": S, "hidden": HIDDEN, "heads": HEADS, "head_dim": HEAD_DIM,
            "intermediate": INTER, "vocab": VOCAB, "ignore_frac": 0.10, "eps": EPS, "rope_theta": THETA,
            "l2": "inputs larger than L2 (every tensor >= 2*S*4096 bytes; lm_head 1.24 GB)",
            "parallelism": "one GPU; under torchrun, data parallel over tokens (each rank its own S tokens; "
                           "all-reduce of the valid-label count before the linear-CE, of the loss, dW and RMSNorm "
                           "dw after the backward)"}


def algorithmic(S, n_valid=None):
    """Algorithmic bytes (memory-bound kernels) and flops (linear-CE) per call.  The
    linear CE's required flops are 6 * n_valid * H * V: a token whose label is
    ignored needs no logits and adds nothing to dX or dW (its dX row is 0), and the
    call computes none for it; 6 * S * H * V is also given, as all_tokens."""
    e = 2
    n_valid = S if n_valid is None else n_valid
    SH, SI = S * HIDDEN, S * INTER
    qk = 2 * S * HEADS * HEAD_DIM
    return {
        "rmsnorm_fwd": 2 * SH * e + S * 4 + HIDDEN * e,
        "rmsnorm_bwd": 3 * SH * e + S * 4 + 2 * HIDDEN * e,
        "rope_fwd": 2 * qk * e,
        "rope_bwd": 2 * qk * e,
        "swiglu_fwd": 3 * SI * e,
        "swiglu_bwd": 5 * SI * e,
        "linear_ce_flops": 6 * n_valid * HIDDEN * VOCAB,
        "linear_ce_flops_all_tokens": 6 * S * HIDDEN * VOCAB,
    }


def gen_inputs(S, seed_offset=0):
    """Host inputs (numpy storage arrays; bf16 as uint16 bits)."""
    from datagen import workloads
    w = workloads.qwen_chain(S)
    if seed_offset:
        for v in w.values():
            v.seed += 1000 * seed_offset
    r, p, s, c = w["rmsnorm"], w["rope"], w["swiglu"], w["linear_ce"]
    return {"x": r.make("x"), "w": r.make("w"), "dy_r": r.make("dy"),
            "q": p.make("q"), "k": p.make("k"), "dq": p.make("dq"), "dk": p.make("dk"),
            "gate": s.make("gate"), "up": s.make("up"), "dy_s": s.make("dy"),
            "X": c.make("X"), "W": c.make("W"), "labels": c.make("labels")}


def to_torch(a, device=None, pin=False):
    import torch
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    if pin:
        return t.pin_memory()
    return t.to(device) if device is not None else t


class Chain:
    """Device buffers of one chain and the calls of one step."""

    def __init__(self, L, inputs, device, dp: DataParallel | None = None):
        import torch
        self.L = L
        self.dp = dp
        bf = torch.bfloat16
        S = inputs["x"].shape[0]
        self.S = S
        self.n_valid = int((inputs["labels"] != -100).sum())
        self.inp = {k: (to_torch(v, device) if v is not None else None) for k, v in inputs.items()}
        self.y = torch.empty(S, HIDDEN, dtype=bf, device=device)
        self.rstd = torch.empty(S, dtype=torch.float32, device=device)
        self.dx = torch.empty(S, HIDDEN, dtype=bf, device=device)
        self.dw = torch.empty(HIDDEN, dtype=bf, device=device)
        self.ws_r = torch.empty(L.liger_rmsnorm_bwd_workspace(S, HIDDEN), dtype=torch.uint8, device=device)
        self.ys = torch.empty(S, INTER, dtype=bf, device=device)
        self.dg = torch.empty(S, INTER, dtype=bf, device=device)
        self.du = torch.empty(S, INTER, dtype=bf, device=device)
        self.loss = torch.empty(1, dtype=torch.float32, device=device)
        self.dX = torch.empty(S, HIDDEN, dtype=bf, device=device)
        self.dW = torch.empty(VOCAB, HIDDEN, dtype=bf, device=device)
        self.ws_c = torch.empty(L.liger_linear_ce_workspace(S, HIDDEN, VOCAB, 0, L.LIGER_BF16), dtype=torch.uint8,
                                device=device)

    def launches_per_step(self):
        # the linear CE runs its GEMMs on the tokens that are not ignored (when some are),
        # after 4 launches that compact them (count, scan, index, gather) and before 2 that
        # put dX, lse and the loss terms back
        S = self.S
        nv = getattr(self, "n_valid", S)
        T = nv if 0 < nv < S else S
        compaction = 6 if 0 < nv < S else 0
        chunk = min(T, 8192, max(128, (T + 1) // 2))
        if chunk >= 1024:
            chunk = min(8192, -(-chunk // 256) * 256)
        chunk = min(chunk, T)
        nchunks = -(-T // chunk)
        # the logits GEMM runs over at most 32 MiB of X rows per launch (4096 rows at hidden 4096)
        sub = max(1, min(chunk, max(256, (32 << 20) // (2 * HIDDEN) // 256 * 256)))
        logits = sum(-(-min(chunk, T - c * chunk) // sub) for c in range(nchunks))
        # the dX GEMM runs over vocabulary slabs of at most 65536 rows
        dx = 1 if VOCAB <= 65536 else -(-VOCAB // 65536)
        # linear CE: label scan, label sort and start tables (once), the logits GEMM launches, per
        # chunk dlogits, the dX GEMM launches and the dW GEMM, loss reduction
        return 1 + 1 + 1 + (1 + 2 + logits + (2 + dx) * nchunks + 1 + compaction) + 1 + 1 + 2

    # the per-step inputs each operator reads first, in the order the step reads them
    FIRST_READS = (("rmsnorm_fwd", ("x",)), ("rope_fwd", ("q", "k")), ("swiglu_fwd", ("gate", "up")),
                   ("linear_ce", ("X", "labels")), ("swiglu_bwd", ("dy_s",)), ("rope_bwd", ("dq", "dk")),
                   ("rmsnorm_bwd", ("dy_r",)))

    def step(self, ev=None, ready=None):
        """One pass of every operator; ev: dict name -> list of (start, end) events;
        ready(input name): makes the stream wait until that input is on the device
        (called before the first operator that reads it)."""
        L, i = self.L, self.inp
        first = dict(self.FIRST_READS)

        def rec(name, fn):
            if ready is not None:
                for k in first[name]:
                    ready(k)
            if ev is None:
                fn()
                return
            import torch
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            ev.setdefault(name, []).append((a, b))

        rec("rmsnorm_fwd", lambda: L.liger_rmsnorm_fwd(i["x"], i["w"], self.y, self.rstd, EPS))
        rec("rope_fwd", lambda: L.liger_rope_fwd(i["q"], i["k"], None, THETA))
        rec("swiglu_fwd", lambda: L.liger_swiglu_fwd(i["gate"], i["up"], self.ys))
        if self.dp is None:
            rec("linear_ce", lambda: L.liger_linear_ce_fwd_bwd(i["X"], i["W"], i["labels"], self.loss, self.dX,
                                                               self.dW, self.ws_c))
        else:
            # data parallel: the mean over every rank's valid tokens
            n = self.dp.valid_count()
            rec("linear_ce", lambda: L.liger_linear_ce_fwd_bwd(i["X"], i["W"], i["labels"], self.loss, self.dX,
                                                               self.dW, self.ws_c, reduction="sum",
                                                               grad_scale=1.0 / max(n, 1)))
        rec("swiglu_bwd", lambda: L.liger_swiglu_bwd(i["dy_s"], i["gate"], i["up"], self.dg, self.du))
        rec("rope_bwd", lambda: L.liger_rope_bwd(i["dq"], i["dk"], None, THETA))
        rec("rmsnorm_bwd", lambda: L.liger_rmsnorm_bwd(i["dy_r"], i["x"], i["w"], self.rstd, self.dx, self.dw,
                                                       self.ws_r))
        if self.dp is not None:
            self.dp.reduce_grads(self.loss, self.dW, self.dw)


def isolated_times(chain, dev):
    """Each memory-bound operator of the chain timed alone: median ms per call
    (timed_median).  Before each launch L2 is flushed by writing a 512 MB buffer
    and then reading it back, so that none of the operator's inputs is resident
    and no other buffer's dirty lines are left for the operator to write back
    (the state ncu's cache control leaves before a capture); the in-place RoPE
    gets its inputs restored first."""
    L, i = chain.L, chain.inp
    flush_l2 = L2Flush(dev)

    ops = {
        "rmsnorm_fwd": lambda: L.liger_rmsnorm_fwd(i["x"], i["w"], chain.y, chain.rstd, EPS),
        "rmsnorm_bwd": lambda: L.liger_rmsnorm_bwd(i["dy_r"], i["x"], i["w"], chain.rstd, chain.dx, chain.dw,
                                                   chain.ws_r),
        "rope_fwd": lambda: L.liger_rope_fwd(i["q"], i["k"], None, THETA),
        "rope_bwd": lambda: L.liger_rope_bwd(i["dq"], i["dk"], None, THETA),
        "swiglu_fwd": lambda: L.liger_swiglu_fwd(i["gate"], i["up"], chain.ys),
        "swiglu_bwd": lambda: L.liger_swiglu_bwd(i["dy_s"], i["gate"], i["up"], chain.dg, chain.du),
    }
    # RoPE rotates in place: each timed call starts from the same values, restored
    # (then the flush) before it, outside the timed region
    saved = {k: i[k].clone() for k in ("q", "k", "dq", "dk")}

    def restore(keys):
        def pre():
            for k in keys:
                i[k].copy_(saved[k])
            flush_l2()
        return pre

    pres = {"rope_fwd": restore(("q", "k")), "rope_bwd": restore(("dq", "dk"))}
    out = {name: timed_median(fn, pre=pres.get(name, flush_l2)) for name, fn in ops.items()}
    for k, v in saved.items():
        i[k].copy_(v)
    del flush_l2, saved
    return out


def fused_linear_swiglu_measure(L, dev, T=8192, H=HIDDEN, I=INTER):
    """FusedLinearSwiGLU at the pages' MLP shape (8192 tokens, hidden 4096,
    intermediate 11008), forward and backward alone: ms and TFLOP/s of the
    operator's useful flops (forward 4*T*H*I; backward 8*T*H*I: dX, dW_g, dW_u;
    the recomputing backward also executes the forward's 4*T*H*I again)."""
    import torch
    from datagen import normal
    X = to_torch(normal(5, "mlp.X", (T, H), "bf16"), dev)
    Wg = to_torch(normal(5, "mlp.Wg", (I, H), "bf16", 0.0, 0.02), dev)
    Wu = to_torch(normal(5, "mlp.Wu", (I, H), "bf16", 0.0, 0.02), dev)
    dH = to_torch(normal(5, "mlp.dH", (T, I), "bf16"), dev)
    out = torch.empty(T, I, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(L.liger_fused_linear_swiglu_workspace(T, I), dtype=torch.uint8, device=dev)
    dX, dWg, dWu = torch.empty_like(X), torch.empty_like(Wg), torch.empty_like(Wu)
    res = {}
    for name, fn, fl in (("fwd", lambda: L.liger_fused_linear_swiglu_fwd(X, Wg, Wu, out), 4 * T * H * I),
                         ("bwd", lambda: L.liger_fused_linear_swiglu_bwd(X, Wg, Wu, dH, dX, dWg, dWu, ws),
                          8 * T * H * I)):
        ms = timed_median(fn)
        res[name] = {"ms": round(ms, 3), "tflops": round(fl / ms / 1e9, 1)}
    res["bwd"]["tflops_executed_12thi"] = round(12 * T * H * I / res["bwd"]["ms"] / 1e9, 1)
    # the same work in native PyTorch (two cuBLAS matmuls, silu * mul; backward by autograd),
    # the comparison the pages quote for this fusion
    import torch.nn.functional as F
    Xr, Gr, Ur = X.detach().clone(), Wg.detach().clone(), Wu.detach().clone()

    def torch_fwd():
        with torch.no_grad():
            return F.silu(Xr @ Gr.t()) * (Xr @ Ur.t())

    def torch_fwd_bwd():
        xs, gs, us = Xr.requires_grad_(True), Gr.requires_grad_(True), Ur.requires_grad_(True)
        h = F.silu(xs @ gs.t()) * (xs @ us.t())
        h.backward(dH)
        xs.grad = gs.grad = us.grad = None

    # the saving pair: the forward also keeps g and u, the backward does not recompute them
    gs_, us_ = torch.empty_like(out), torch.empty_like(out)
    res["fwd_save_ms"] = round(timed_median(lambda: L.liger_fused_linear_swiglu_fwd_save(X, Wg, Wu, out, gs_, us_)), 3)
    res["bwd_saved_ms"] = round(timed_median(
        lambda: L.liger_fused_linear_swiglu_bwd_saved(X, Wg, Wu, dH, gs_, us_, dX, dWg, dWu, ws)), 3)
    t_fwd = timed_median(torch_fwd)
    t_fb = timed_median(torch_fwd_bwd)
    res["torch_fwd_ms"] = round(t_fwd, 3)
    res["torch_bwd_ms"] = round(max(t_fb - t_fwd, 1e-6), 3)
    res["speedup_fwd_vs_torch"] = round(t_fwd / res["fwd"]["ms"], 3)
    res["speedup_bwd_vs_torch"] = round(res["torch_bwd_ms"] / res["bwd"]["ms"], 3)
    res["speedup_fwd_bwd_vs_torch"] = round(t_fb / (res["fwd"]["ms"] + res["bwd"]["ms"]), 3)
    res["speedup_fwd_bwd_saved_vs_torch"] = round(t_fb / (res["fwd_save_ms"] + res["bwd_saved_ms"]), 3)
    # the training pair (the forward keeps g and u for the backward, as autograd keeps its activations)
    fb = res["fwd_save_ms"] + res["bwd_saved_ms"]
    res["fwd_bwd"] = {"pair": "liger_fused_linear_swiglu_fwd_save + liger_fused_linear_swiglu_bwd_saved",
                      "ms": round(fb, 3), "tflops": round(12 * T * H * I / fb / 1e9, 1),
                      "torch_ms": round(t_fb, 3), "speedup_vs_torch": round(t_fb / fb, 3)}
    return res


WARMUP_ITERS, MIN_ITERS, MIN_TIMED_MS, FLOOR_ITERS = 10, 50, 200.0, 5
# DRAM bytes (read + written) of one linear-CE call at seq 32768 with 10 % of the labels ignored
# (29491 valid tokens: compaction, then chunks of 8192, 8192, 8192 and 4915 rows): the sum of
# ncu's dram__bytes_read.sum + dram__bytes_write.sum over the 38 launches of one whole call
LINEAR_CE_TRAFFIC = 144_775_323_904


def linear_ce_algorithmic_bytes(n_valid, T, H=None, V=None, chunk=8192):
    """The bytes a token-chunked linear-CE call must move at least, each tensor once per pass
    that has to touch it: per valid token 10*V bytes of the bf16 chunk buffer (P written,
    dlogits reading P and writing D, the dX and dW GEMMs reading D), W read twice per chunk
    (logits, dX), the fp32 dW sum written by every chunk but the last and read by every
    chunk but the first, the bf16 dW written once, the compacted X rows read twice (logits,
    dW) and dX rows written once, and the compaction's gather (valid X rows read and
    written) and scatter (valid dX rows read, all T dX rows written)."""
    H = HIDDEN if H is None else H
    V = VOCAB if V is None else V
    nchunks = -(-n_valid // chunk)
    b = 10 * n_valid * V + 2 * nchunks * V * H * 2 + 2 * max(0, nchunks - 1) * V * H * 4 + V * H * 2
    b += 3 * n_valid * H * 2
    if n_valid < T:
        b += 2 * n_valid * H * 2 + n_valid * H * 2 + T * H * 2
    return b


def timed_median(fn, pre=None):
    """Median ms of one call of fn, timed with CUDA events on the current
    stream: 10 untimed warm-up calls, then timed calls until 50 have run or
    200 ms have been timed (and at least 5 have run).  pre() runs before every
    call, outside the timed region (the L2 flush of the memory-bound ops)."""
    import torch
    for _ in range(WARMUP_ITERS):
        if pre is not None:
            pre()
        fn()
    torch.cuda.synchronize()
    ts = []
    while len(ts) < MIN_ITERS and not (sum(ts) >= MIN_TIMED_MS and len(ts) >= FLOOR_ITERS):
        if pre is not None:
            pre()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def rmsnorm_qkv_rope_measure(L, dev, S=32768, H=HIDDEN, Hq=HEADS, Hk=HEADS, D=HEAD_DIM):
    """Fused RMSNorm + QKV projection (+ bias) + RoPE forward at the Qwen-7B layer
    shapes and the chain's sequence length, alone: the whole call (weight fold,
    rstd/angle pre-pass, GEMM with the scale/bias/RoPE epilogue), the call with
    the folded weights reused, and for comparison the unfused sequence of the
    same work (RMSNorm kernel, cuBLAS addmm with the bias, RoPE kernel on the
    packed QKV views).  2*T*H*N flops, N = (Hq + 2 Hk) D."""
    import torch
    from datagen import normal
    T, nq, nk = S, Hq * D, Hk * D
    N = nq + 2 * nk
    x = to_torch(normal(6, "qkv.x", (T, H), "bf16"), dev)
    wn = to_torch(normal(6, "qkv.w", (H,), "bf16", 1.0, 0.1), dev)
    Wq = to_torch(normal(6, "qkv.Wq", (nq, H), "bf16", 0.0, 0.02), dev)
    Wk = to_torch(normal(6, "qkv.Wk", (nk, H), "bf16", 0.0, 0.02), dev)
    Wv = to_torch(normal(6, "qkv.Wv", (nk, H), "bf16", 0.0, 0.02), dev)
    bq = to_torch(normal(6, "qkv.bq", (nq,), "bf16", 0.0, 0.1), dev)
    bk = to_torch(normal(6, "qkv.bk", (nk,), "bf16", 0.0, 0.1), dev)
    bv = to_torch(normal(6, "qkv.bv", (nk,), "bf16", 0.0, 0.1), dev)
    q = torch.empty(1, S, Hq, D, dtype=torch.bfloat16, device=dev)
    k = torch.empty(1, S, Hk, D, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    ws = torch.empty(L.liger_rmsnorm_qkv_rope_workspace(T, H, Hq, Hk, D), dtype=torch.uint8, device=dev)
    fl = 2.0 * T * H * N

    def fused(folded):
        return lambda: L.liger_rmsnorm_qkv_rope_fwd(x, wn, Wq, Wk, Wv, q, k, v, ws, 1, S, Hq, Hk, D, bq=bq, bk=bk,
                                                    bv=bv, eps=EPS, theta=THETA, folded=folded)

    ms_full = timed_median(fused(False))
    ms_folded = timed_median(fused(True))
    del ws
    Wcat = torch.cat([Wq, Wk, Wv]).t()
    bcat = torch.cat([bq, bk, bv])
    xn = torch.empty_like(x)
    qkv = torch.empty(T, N, dtype=torch.bfloat16, device=dev)

    def unfused():
        L.liger_rmsnorm_fwd(x, wn, xn, None, EPS)
        torch.addmm(bcat, xn, Wcat, out=qkv)
        L.liger_rope_fwd_ex(qkv, qkv[:, nq:], N, N, Hq, Hk, D, 1, S, theta=THETA)

    ms_unf = timed_median(unfused)
    return {"ms": round(ms_full, 3), "tflops": round(fl / ms_full / 1e9, 1),
            "ms_folded_weights": round(ms_folded, 3), "tflops_folded_weights": round(fl / ms_folded / 1e9, 1),
            "ms_unfused_cublas": round(ms_unf, 3), "speedup_vs_unfused": round(ms_unf / ms_full, 3)}


def linear_ce_two_pass_measure(chain, dev):
    """The two-pass, vocabulary-chunked linear CE on the chain's own head inputs
    (seq x 4096 x 151936, 10 % of labels ignored), alone: ms, TFLOP/s of the
    operator's useful 6*n_valid*H*V flops and of the 8*n_valid*H*V it executes
    (the logits twice; the ignored tokens are not run), and both variants'
    workspace bytes."""
    import torch
    L, i, S = chain.L, chain.inp, chain.S
    ws = torch.empty(L.liger_linear_ce_two_pass_workspace(S, HIDDEN, VOCAB), dtype=torch.uint8, device=dev)
    ms = timed_median(lambda: L.liger_linear_ce_two_pass_fwd_bwd(i["X"], i["W"], i["labels"], chain.loss, chain.dX,
                                                               chain.dW, ws))
    fl = float(chain.n_valid) * HIDDEN * VOCAB
    return {"ms": round(ms, 3), "n_valid": chain.n_valid, "tflops_8nhv": round(8 * fl / ms / 1e9, 1),
            "tflops_6nhv": round(6 * fl / ms / 1e9, 1),
            "workspace_bytes": int(ws.numel()), "workspace_bytes_token_chunked": int(chain.ws_c.numel())}


# ------------------------------------------------------- named workloads
class L2Flush:
    """Writes a 512 MB buffer and reads it back: afterwards no input of the next
    call is resident in the 129 MB L2 and no other buffer's dirty lines are
    left for the call to write back."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        import torch
        self.buf.zero_()
        self.buf.view(torch.int32).amax()


def _hbm_entry(nbytes, ms, pk):
    gbs = nbytes / (ms / 1000.0) / 1e9
    return {"ms": round(ms, 4), "bytes": int(nbytes), "gbs": round(gbs, 1), "frac": round(gbs / pk["hbm_gbs"], 4)}


def tiny_latency(L, dev, flush):
    """The tiny decoder-op set (batch 2, seq 128, hidden 256, 4 heads x 64,
    intermediate 688, vocab 1024) in fp32 and bf16: median latency of each
    operator call in microseconds, L2 flushed before every call (the set fits
    in L2).  fp32 linear-CE runs on the fp32 SIMT path, bf16 on the tensor cores."""
    import torch
    from datagen import workloads
    out = {}
    for dt in ("f32", "bf16"):
        w = workloads.tiny(dt)
        r, p, sw, c = w["rmsnorm"], w["rope"], w["swiglu"], w["linear_ce"]
        x, wn, dy = (to_torch(r.make(k), dev) for k in ("x", "w", "dy"))
        q, k = to_torch(p.make("q"), dev), to_torch(p.make("k"), dev)
        g, u, dys = (to_torch(sw.make(k_), dev) for k_ in ("gate", "up", "dy"))
        X, W = to_torch(c.make("X"), dev), to_torch(c.make("W"), dev)
        lab = torch.from_numpy(c.make("labels")).to(dev)
        T, H = x.shape
        y, dx, dw = torch.empty_like(x), torch.empty_like(x), torch.empty_like(wn)
        rstd = torch.empty(T, dtype=torch.float32, device=dev)
        wsr = torch.empty(L.liger_rmsnorm_bwd_workspace(T, H), dtype=torch.uint8, device=dev)
        ys, dg, du = torch.empty_like(g), torch.empty_like(g), torch.empty_like(g)
        loss = torch.empty(1, dtype=torch.float32, device=dev)
        dX, dW = torch.empty_like(X), torch.empty_like(W)
        code = L.LIGER_F32 if dt == "f32" else L.LIGER_BF16
        wsc = torch.empty(L.liger_linear_ce_workspace(T, H, W.shape[0], 0, code), dtype=torch.uint8, device=dev)
        eps, theta = r.params["eps"], p.params["theta"]
        L.liger_rmsnorm_fwd(x, wn, y, rstd, eps)
        ops = {
            "rmsnorm_fwd": lambda: L.liger_rmsnorm_fwd(x, wn, y, rstd, eps),
            "rmsnorm_bwd": lambda: L.liger_rmsnorm_bwd(dy, x, wn, rstd, dx, dw, wsr),
            "rope_fwd": lambda: L.liger_rope_fwd(q, k, None, theta),
            "rope_bwd": lambda: L.liger_rope_bwd(q, k, None, theta),
            "swiglu_fwd": lambda: L.liger_swiglu_fwd(g, u, ys),
            "swiglu_bwd": lambda: L.liger_swiglu_bwd(dys, g, u, dg, du),
            "linear_ce_fwd_bwd": lambda: L.liger_linear_ce_fwd_bwd(X, W, lab, loss, dX, dW, wsc),
        }
        out[dt] = {name: round(1000.0 * timed_median(fn, pre=flush), 2) for name, fn in ops.items()}
    out["unit"] = "us per call (median, L2 flushed before each call)"
    out["shape"] = "T=256 H=256 heads 4x64 I=688 V=1024"
    return out


def swiglu_config(L, dev, flush, pk):
    """SwiGLU fwd and bwd on gate/up [4, 2048, 11008] bf16 (seed 1), alone, L2
    flushed before each call: 3 and 5 bytes x 2 per element."""
    import torch
    from datagen import workloads
    w = workloads.swiglu_llama()
    g, u, dy = (to_torch(w.make(k), dev) for k in ("gate", "up", "dy"))
    y, dg, du = torch.empty_like(g), torch.empty_like(g), torch.empty_like(g)
    n = g.numel()
    f = timed_median(lambda: L.liger_swiglu_fwd(g, u, y), pre=flush)
    b = timed_median(lambda: L.liger_swiglu_bwd(dy, g, u, dg, du), pre=flush)
    return {"shape": "gate/up [4,2048,11008] bf16", "fwd": _hbm_entry(3 * n * 2, f, pk),
            "bwd": _hbm_entry(5 * n * 2, b, pk)}


def llama3_norm_rope_config(L, dev, flush, pk):
    """RMSNorm fwd/bwd on x [32768, 4096] (eps 1e-5) and RoPE fwd/bwd on
    Q [4, 8192, 32, 128] + K [4, 8192, 8, 128] (theta 5e5), bf16, seed 2,
    alone, L2 flushed before each call (RoPE's inputs restored first)."""
    import torch
    from datagen import workloads
    w = workloads.rmsnorm_rope_llama3()
    r, p = w["rmsnorm"], w["rope"]
    x, wn, dy = (to_torch(r.make(k), dev) for k in ("x", "w", "dy"))
    T, H = x.shape
    y, dx, dw = torch.empty_like(x), torch.empty_like(x), torch.empty_like(wn)
    rstd = torch.empty(T, dtype=torch.float32, device=dev)
    wsr = torch.empty(L.liger_rmsnorm_bwd_workspace(T, H), dtype=torch.uint8, device=dev)
    eps, theta = r.params["eps"], p.params["theta"]
    L.liger_rmsnorm_fwd(x, wn, y, rstd, eps)
    rf = timed_median(lambda: L.liger_rmsnorm_fwd(x, wn, y, rstd, eps), pre=flush)
    rb = timed_median(lambda: L.liger_rmsnorm_bwd(dy, x, wn, rstd, dx, dw, wsr), pre=flush)
    del y, dx
    q, k, dq, dk = (to_torch(p.make(n), dev) for n in ("q", "k", "dq", "dk"))
    saved = {n: t.clone() for n, t in (("q", q), ("k", k), ("dq", dq), ("dk", dk))}

    def restore(*pairs):
        def pre():
            for t, n in pairs:
                t.copy_(saved[n])
            flush()
        return pre
    pf = timed_median(lambda: L.liger_rope_fwd(q, k, None, theta), pre=restore((q, "q"), (k, "k")))
    pb = timed_median(lambda: L.liger_rope_bwd(dq, dk, None, theta), pre=restore((dq, "dq"), (dk, "dk")))
    e = 2
    qk = q.numel() + k.numel()
    return {"shape": "x [32768,4096]; Q [4,8192,32,128] + K [4,8192,8,128] theta 5e5, bf16",
            "rmsnorm_fwd": _hbm_entry(2 * T * H * e + 4 * T + H * e, rf, pk),
            "rmsnorm_bwd": _hbm_entry(3 * T * H * e + 4 * T + 2 * H * e, rb, pk),
            "rope_fwd": _hbm_entry(2 * qk * e, pf, pk), "rope_bwd": _hbm_entry(2 * qk * e, pb, pk)}


def llama3_head_config(L, dev, pk):
    """Fused linear-CE fwd+bwd at the Llama-3 head: 8192 tokens x hidden 4096 x
    vocab 128256 bf16, 10 % ignored labels, mean (seed 3), back-to-back calls
    (lm_head 1.05 GB: larger than L2).  6*n_valid*H*V required flops per call."""
    import torch
    from datagen import workloads
    c = workloads.linear_ce_llama3()
    X, W = to_torch(c.make("X"), dev), to_torch(c.make("W"), dev)
    lab = torch.from_numpy(c.make("labels")).to(dev)
    T, H = X.shape
    V = W.shape[0]
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    dX, dW = torch.empty_like(X), torch.empty_like(W)
    ws = torch.empty(L.liger_linear_ce_workspace(T, H, V, 0, L.LIGER_BF16), dtype=torch.uint8, device=dev)
    ms = timed_median(lambda: L.liger_linear_ce_fwd_bwd(X, W, lab, loss, dX, dW, ws))
    n_valid = int((lab != -100).sum().item())
    tf = 6.0 * n_valid * H * V / (ms / 1000.0) / 1e12
    return {"shape": "T=8192 H=4096 V=128256 bf16, mean, 10% ignored", "ms": round(ms, 3),
            "tokens_per_s": round(T / (ms / 1000.0), 1), "n_valid": n_valid,
            "tflops_6nhv": round(tf, 1), "tflops_counting_all_tokens": round(6.0 * T * H * V / (ms / 1000.0) / 1e12, 1),
            "frac_sustained": round(tf / pk["bf16_sustained"], 4), "frac_burst": round(tf / pk["bf16"], 4),
            "loss": float(loss.item()),
            "timing": "median of >= 50 back-to-back calls after 10 warm-ups (power-capped clock: compare with "
                      "the sustained peak)"}


def chain_sweep(L, dev, flush, base_inputs, seqs=(512, 2048, 8192), steps=10):
    """The layer chain at shorter sequences (the same named tensors of seed 4,
    i.e. the first S rows of the seq-32768 draws, and labels drawn for S
    tokens): median ms of one step (every operator fwd+bwd) with L2 flushed
    before each step, and tokens/s = S / that time."""
    import torch
    from datagen import workloads
    out = {}
    for S in seqs:
        inp = {}
        for k_, v in base_inputs.items():
            if k_ in ("q", "k", "dq", "dk"):
                inp[k_] = np.ascontiguousarray(v[:, :S])
            elif k_ in ("w", "W"):
                inp[k_] = v
            elif k_ == "labels":
                inp[k_] = workloads.qwen_chain(S)["linear_ce"].make("labels")
            else:
                inp[k_] = np.ascontiguousarray(v[:S])
        ch = Chain(L, inp, dev)
        for _ in range(3):
            ch.step()
        ts = []
        for _ in range(steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            ch.step()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        out[str(S)] = {"ms_per_step": round(ms, 3), "tokens_per_s": round(S / (ms / 1000.0), 1)}
        del ch
        torch.cuda.empty_cache()
    out["timing"] = f"median of {steps} steps, L2 flushed before each"
    return out


def named_configs(L, dev, pk, chain_inputs):
    flush = L2Flush(dev)
    res = {"tiny_set": tiny_latency(L, dev, flush),
           "swiglu_4x2048x11008": swiglu_config(L, dev, flush, pk),
           "llama3_rmsnorm_rope": llama3_norm_rope_config(L, dev, flush, pk),
           "llama3_linear_ce": llama3_head_config(L, dev, pk),
           "qwen_chain_seq_sweep": chain_sweep(L, dev, flush, chain_inputs)}
    del flush
    return res


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.idx = gpu_index
        # the raw samples go to $BENCH_CLOCKS_DIR (default: the system temporary directory)
        import tempfile
        self.path = os.path.join(os.environ.get("BENCH_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
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
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = max(mx, float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return None
        loaded = [x for x in sm if x > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- CPU oracle
def cpu_oracle_sample(S, inputs, n_rows=32, n_tokens=1):
    """Time the fp64 oracle (single-threaded) on a bounded sample of the
    chain's workload; returns (tokens/s, description, seconds)."""
    import oracle
    r = np.random.default_rng(0).choice(S, n_rows, replace=False)
    x, w, dy = inputs["x"][r], inputs["w"], inputs["dy_r"][r]
    per_token = 0.0
    t0 = time.perf_counter()
    oracle.rmsnorm_fwd(x, w, EPS)
    oracle.rmsnorm_bwd(dy, x, w, EPS)
    per_token += (time.perf_counter() - t0) / n_rows
    q = np.ascontiguousarray(inputs["q"][:, r]); k = np.ascontiguousarray(inputs["k"][:, r])
    pos = r.astype(np.int32)[None, :]
    t0 = time.perf_counter()
    oracle.rope(q, THETA, pos=pos); oracle.rope(k, THETA, pos=pos)
    oracle.rope(q, THETA, sign=-1, pos=pos); oracle.rope(k, THETA, sign=-1, pos=pos)
    per_token += (time.perf_counter() - t0) / n_rows
    g, u, ds = inputs["gate"][r], inputs["up"][r], inputs["dy_s"][r]
    t0 = time.perf_counter()
    oracle.swiglu_fwd(g, u)
    oracle.swiglu_bwd(ds, g, u)
    per_token += (time.perf_counter() - t0) / n_rows
    lab = inputs["labels"]
    valid = np.nonzero(lab != -100)[0][:n_tokens]
    X = np.ascontiguousarray(inputs["X"][valid])
    t0 = time.perf_counter()
    oracle.linear_ce(X, inputs["W"], lab[valid])
    per_token += (time.perf_counter() - t0) / len(valid)
    desc = (f"fp64 oracle, 1 thread: RMSNorm/RoPE/SwiGLU fwd+bwd on {n_rows} random rows/positions of seq {S}, "
            f"linear-CE fwd+bwd (lse, dX, dW) on {len(valid)} token(s) x full vocab {VOCAB}; tokens/s = 1 / sum of "
            f"per-token times")
    return 1.0 / per_token, desc, per_token


# Arm CPU parts by (implementer, part) of the main ID register, as /proc/cpuinfo prints them
ARM_PARTS = {("0x41", "0xd4f"): "Arm Neoverse V2", ("0x41", "0xd40"): "Arm Neoverse V1",
             ("0x41", "0xd0c"): "Arm Neoverse N1", ("0x41", "0xd49"): "Arm Neoverse N2",
             ("0x41", "0xd84"): "Arm Neoverse V3", ("0x41", "0xd8e"): "Arm Neoverse N3"}


def cpu_model(cpuinfo_text: str, lscpu_text: str = "") -> str | None:
    """The CPU model: /proc/cpuinfo's model name (x86), else lscpu's "Model
    name", else the Arm implementer/part pair of /proc/cpuinfo, named where known."""
    for line in cpuinfo_text.splitlines():
        k, _, v = line.partition(":")
        if k.strip().lower() in ("model name", "cpu model", "processor name") and v.strip():
            return v.strip()
    for line in lscpu_text.splitlines():
        k, _, v = line.partition(":")
        if k.strip().lower() == "model name" and v.strip() and v.strip() != "-":
            return v.strip()
    impl = part = None
    for line in cpuinfo_text.splitlines():
        k, _, v = line.partition(":")
        k, v = k.strip().lower(), v.strip().lower()
        if k == "cpu implementer" and impl is None:
            impl = v
        elif k == "cpu part" and part is None:
            part = v
    if impl and part:
        name = ARM_PARTS.get((impl, part))
        return f"{name} (implementer {impl}, part {part})" if name else f"Arm implementer {impl}, part {part}"
    return None


def host_cpu():
    """The host the oracle ran on: logical CPUs and the CPU model."""
    import platform
    info = ls = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        pass
    try:
        ls = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
    except Exception:
        pass
    return {"host_nproc": os.cpu_count(), "host_cpu": cpu_model(info, ls) or platform.machine(),
            "host_arch": platform.machine()}


def emit(d):
    print(json.dumps(d), flush=True)


# ---------------------------------------------------------------- arms
def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    S = args.seq
    inputs = gen_inputs(S)
    vals = []
    for i in range(args.warmup + args.steps):
        v, desc, _ = cpu_oracle_sample(S, inputs, n_rows=16, n_tokens=1)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.mean(vals)
    d = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
         "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * S / value,
         "ms_per_step_kind": f"extrapolated: seq {S} tokens / the tokens/s of a 16-row / 1-token sample per step",
         "higher_is_better": True,
         "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": workload_config(S),
         "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc, **host_cpu()},
         "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    emit(d)
    return 0


def native_arm(args):
    import torch
    rank, world, local = dist_env()
    dist = dist_init(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import transformer_rmsnorm_fwd_gb300 as L
    L.load()
    S, K, W = args.seq, args.steps, args.warmup
    assert W >= 0 and K >= 1
    inputs = gen_inputs(S, seed_offset=rank)
    dp = DataParallel(dist, int((inputs["labels"] != -100).sum()), dev) if dist else None
    chain = Chain(L, inputs, dev, dp)
    torch.cuda.synchronize()

    # ---- device-resident timing
    for _ in range(W):
        chain.step()
    ev = {}
    clk = ClockSampler(local)
    clk.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record()
    for _ in range(K):
        chain.step(ev)
    t_end.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = clk.stop()
    ms = max_over_ranks(t_start.elapsed_time(t_end), dist, dev)
    tokens = sum_over_ranks(float(S * K), dist, dev)
    value = tokens / (ms / 1000.0)
    per_op = {k: sum(a.elapsed_time(b) for a, b in v) / len(v) for k, v in ev.items()}
    loss = float(chain.loss.item())
    if dp is not None:
        loss = dp.mean_loss(loss)

    # ---- end to end through host buffers (measured right after the device-resident steps, so
    # that both see the GPU in the same power and thermal state): every step copies its inputs (activations,
    # labels, upstream gradients) host -> device from pinned memory and reads its loss back;
    # the parameters (RMSNorm weight, lm_head weight) stay resident on the device, as in a
    # training loop.  The copies run on a second stream into the other half of a
    # double-buffered input set, overlapping the previous step's kernels; the timed region
    # spans all K steps' copies and kernels.
    e2e = None
    if not args.no_e2e:
        host = {k: to_torch(v, pin=True) for k, v in inputs.items() if k not in PARAMETERS}
        h_loss = torch.empty(K + max(1, W), dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        sets = [chain.inp, {k: (v if k in PARAMETERS else torch.empty_like(v)) for k, v in chain.inp.items()}]
        copy_stream = torch.cuda.Stream(device=dev)
        compute = torch.cuda.current_stream(dev)
        # inputs copied in the order the step first reads them, one event per input, so each
        # operator waits only for its own inputs (the first step of a run starts as soon as x
        # is on the device instead of after all 4 GB)
        order = [k for _, names in Chain.FIRST_READS for k in names]
        assert sorted(order) == sorted(host), (order, sorted(host))
        copied = [{k: torch.cuda.Event() for k in order} for _ in range(2)]
        consumed = [torch.cuda.Event(), torch.cuda.Event()]

        def enqueue_copy(i):
            s = i % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(consumed[s])      # the step that last used this set is done
                for k in order:
                    sets[s][k].copy_(host[k], non_blocking=True)
                    copied[s][k].record(copy_stream)

        def run(n, offset):
            enqueue_copy(0)
            for i in range(n):
                s = i % 2
                if i + 1 < n:
                    enqueue_copy(i + 1)
                chain.inp = sets[s]
                chain.step(ready=lambda k, s=s: compute.wait_event(copied[s][k]))
                consumed[s].record(compute)
                h_loss[offset + i].copy_(chain.loss[0], non_blocking=True)

        for ev in consumed:
            ev.record(compute)
        # the copy alone: one step's inputs host -> device on the copy stream
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(copy_stream):
            c0.record(copy_stream)
            for k, t in host.items():
                sets[1][k].copy_(t, non_blocking=True)
            c1.record(copy_stream)
        torch.cuda.synchronize()
        h2d_ms = c0.elapsed_time(c1)
        run(max(1, W), K)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(compute)
        run(K, 0)
        b.record(compute)
        torch.cuda.synchronize()
        ms_e = max_over_ranks(a.elapsed_time(b), dist, dev)
        e2e = {"value": tokens / (ms_e / 1000.0), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": 4, "ms_per_step": ms_e / K,
               "pipelining": "inputs of step i+1 copied on a second stream during step i (double-buffered), "
                             "each operator waiting only for the inputs it reads",
               "resident": "parameters " + ", ".join(sorted(PARAMETERS)) + " stay on the device",
               "h2d_alone_ms": round(h2d_ms, 3), "h2d_alone_gbs": round(h2d / (h2d_ms / 1000.0) / 1e9, 1)}
        chain.inp = sets[0]
        del host, sets

    # ---- each memory-bound operator alone, and the operators of the next rows
    iso = isolated_times(chain, dev)
    mlp = fused_linear_swiglu_measure(L, dev)
    qkv = rmsnorm_qkv_rope_measure(L, dev, S)
    two_pass = linear_ce_two_pass_measure(chain, dev)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    pk = peaks()
    configs = None
    if not args.no_configs:
        configs = named_configs(L, dev, pk, inputs)
    n_valid = int((inputs["labels"] != -100).sum())
    alg = algorithmic(S, n_valid)
    hbm = {}
    for k in ("rmsnorm_fwd", "rmsnorm_bwd", "rope_fwd", "rope_bwd", "swiglu_fwd", "swiglu_bwd"):
        gbs = alg[k] / (per_op[k] / 1000.0) / 1e9
        gi = alg[k] / (iso[k] / 1000.0) / 1e9
        hbm[k] = {"ms": round(per_op[k], 4), "bytes": alg[k], "gbs": round(gbs, 1),
                  "frac": round(gbs / pk["hbm_gbs"], 4), "ms_isolated": round(iso[k], 4),
                  "gbs_isolated": round(gi, 1), "frac_isolated": round(gi / pk["hbm_gbs"], 4)}
    ce_tf = alg["linear_ce_flops"] / (per_op["linear_ce"] / 1000.0) / 1e12
    roofline = {"kernel": "liger_linear_ce_fwd_bwd (tcgen05 GEMMs + fused epilogues; 6*n_valid*H*V flops per call: "
                          "the ignored tokens' logits are not computed)",
                "bound": "tensor", "achieved": round(ce_tf, 1), "peak": pk["bf16_sustained"], "unit": "TFLOP/s",
                "frac": round(ce_tf / pk["bf16_sustained"], 4), "n_valid": n_valid, "tokens": S,
                "achieved_counting_all_tokens": round(alg["linear_ce_flops_all_tokens"] /
                                                      (per_op["linear_ce"] / 1000.0) / 1e12, 1),
                "traffic": LINEAR_CE_TRAFFIC if S == 32768 else None, "traffic_unit": "bytes per call",
                "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum summed over the 38 launches "
                                  "of one whole call (seq 32768, 29491 valid tokens)",
                "traffic_algorithmic": linear_ce_algorithmic_bytes(n_valid, S),
                "peak_source": f"{pk['src']} bf16 sustained (cuBLAS loop under the power cap)",
                "ms_per_call": round(per_op["linear_ce"], 3)}
    cpu = None
    if not args.no_cpu:
        v, desc, _ = cpu_oracle_sample(S, inputs)
        cpu = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc, **host_cpu()}
    d = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
         "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
         "data": "synthetic (seeded SplitMix64/Box-Muller, shapes and distributions of the Qwen-7B layer chain)",
         "config": workload_config(S), "roofline": roofline, "hbm_kernels": hbm,
         "hbm_peak_gbs": pk["hbm_gbs"], "cpu_baseline": cpu, "e2e": e2e, "configs": configs,
         "gpu_launches": chain.launches_per_step() * K, "clocks": clocks, "loss": loss,
         "fused_linear_swiglu": dict(mlp, shape="T=8192 H=4096 I=11008 bf16 (alone, not part of the step)",
                                     peak_tflops_burst=pk["bf16"], peak_tflops_sustained=pk["bf16_sustained"],
                                     flops="useful: fwd 4*T*H*I, bwd 8*T*H*I, fwd_bwd 12*T*H*I",
                                     frac_fwd=round(mlp["fwd"]["tflops"] / pk["bf16"], 4),
                                     frac_bwd=round(mlp["bwd"]["tflops"] / pk["bf16"], 4),
                                     frac_fwd_sustained=round(mlp["fwd"]["tflops"] / pk["bf16_sustained"], 4),
                                     frac_bwd_sustained=round(mlp["bwd"]["tflops"] / pk["bf16_sustained"], 4),
                                     frac_fwd_bwd_sustained=round(mlp["fwd_bwd"]["tflops"] / pk["bf16_sustained"],
                                                                  4),
                                     timing="median of >= 50 back-to-back calls after 10 warm-ups (power-capped "
                                            "clock: compare with the sustained peak)"),
         "rmsnorm_qkv_rope": dict(qkv, shape=f"T={S} H={HIDDEN} Hq=Hk={HEADS} D={HEAD_DIM} QKV bias, bf16 "
                                             "(alone, not part of the step)",
                                  peak_tflops_burst=pk["bf16"], peak_tflops_sustained=pk["bf16_sustained"],
                                  frac=round(qkv["tflops"] / pk["bf16"], 4),
                                  frac_folded_weights=round(qkv["tflops_folded_weights"] / pk["bf16"], 4),
                                  frac_sustained=round(qkv["tflops"] / pk["bf16_sustained"], 4),
                                  frac_folded_weights_sustained=round(qkv["tflops_folded_weights"] /
                                                                      pk["bf16_sustained"], 4),
                                  timing="median of >= 50 back-to-back calls after 10 warm-ups (power-capped "
                                         "clock: compare with the sustained peak)"),
         "linear_ce_two_pass": dict(two_pass, shape=f"S={S} H={HIDDEN} V={VOCAB} bf16, auto vocabulary chunk "
                                                    "(alone, not part of the step)",
                                    frac_useful_6nhv=round(two_pass["tflops_6nhv"] / pk["bf16_sustained"], 4),
                                    frac_executed_8nhv=round(two_pass["tflops_8nhv"] / pk["bf16_sustained"], 4))}
    emit(d)
    if dist:
        dist.destroy_process_group()
    return 0


def single_op(args):
    """One operator alone, W untimed + K timed calls on device-resident inputs
    (the profiling cases: small enough for a few GB on the device)."""
    import torch
    import transformer_rmsnorm_fwd_gb300 as L
    from datagen import labels, normal
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    L.load()
    S, op = args.seq, args.op
    bf = torch.bfloat16
    if op in ("linear_ce", "linear_ce_two_pass"):
        X = to_torch(normal(7, "op.X", (S, HIDDEN), "bf16"), dev)
        W = to_torch(normal(7, "op.W", (VOCAB, HIDDEN), "bf16", 0.0, 0.02), dev)
        lab = torch.from_numpy(labels(7, "op.labels", S, VOCAB, args.ignore_frac)).to(dev)
        loss = torch.empty(1, dtype=torch.float32, device=dev)
        dX, dW = torch.empty_like(X), torch.empty_like(W)
        if op == "linear_ce":
            ws = torch.empty(L.liger_linear_ce_workspace(S, HIDDEN, VOCAB, args.chunk, L.LIGER_BF16),
                             dtype=torch.uint8, device=dev)
            fn = lambda: L.liger_linear_ce_fwd_bwd(X, W, lab, loss, dX, dW, ws, chunk=args.chunk)
            # the GEMMs run on the tokens whose label is not ignored
            flops = 6.0 * int((lab != -100).sum()) * HIDDEN * VOCAB
        else:
            ws = torch.empty(L.liger_linear_ce_two_pass_workspace(S, HIDDEN, VOCAB), dtype=torch.uint8, device=dev)
            fn = lambda: L.liger_linear_ce_two_pass_fwd_bwd(X, W, lab, loss, dX, dW, ws)
            flops = 8.0 * S * HIDDEN * VOCAB
    elif op == "rmsnorm_qkv_rope":
        N = 3 * HEADS * HEAD_DIM
        x = to_torch(normal(7, "op.x", (S, HIDDEN), "bf16"), dev)
        wn = to_torch(normal(7, "op.w", (HIDDEN,), "bf16", 1.0, 0.1), dev)
        Wq, Wk, Wv = (to_torch(normal(7, f"op.W{c}", (HEADS * HEAD_DIM, HIDDEN), "bf16", 0.0, 0.02), dev)
                      for c in "qkv")
        q = torch.empty(1, S, HEADS, HEAD_DIM, dtype=bf, device=dev)
        k, v = torch.empty_like(q), torch.empty_like(q)
        ws = torch.empty(L.liger_rmsnorm_qkv_rope_workspace(S, HIDDEN, HEADS, HEADS, HEAD_DIM), dtype=torch.uint8,
                         device=dev)
        fn = lambda: L.liger_rmsnorm_qkv_rope_fwd(x, wn, Wq, Wk, Wv, q, k, v, ws, 1, S, HEADS, HEADS, HEAD_DIM,
                                                  eps=EPS, theta=THETA)
        flops = 2.0 * S * HIDDEN * N
    elif op in ("rmsnorm", "rope", "swiglu"):
        # forward then backward, HBM-bound: report GB/s of the algorithmic bytes
        e = 2
        if op == "rmsnorm":
            x = to_torch(normal(7, "op.rx", (S, HIDDEN), "bf16"), dev)
            w = to_torch(normal(7, "op.rw", (HIDDEN,), "bf16", 1.0, 0.1), dev)
            dy = to_torch(normal(7, "op.rdy", (S, HIDDEN), "bf16"), dev)
            y, dx, dw = torch.empty_like(x), torch.empty_like(x), torch.empty_like(w)
            rstd = torch.empty(S, dtype=torch.float32, device=dev)
            wsr = torch.empty(L.liger_rmsnorm_bwd_workspace(S, HIDDEN), dtype=torch.uint8, device=dev)

            def fn():
                L.liger_rmsnorm_fwd(x, w, y, rstd, EPS)
                L.liger_rmsnorm_bwd(dy, x, w, rstd, dx, dw, wsr)
            nbytes = (2 * S * HIDDEN * e + 4 * S) + (3 * S * HIDDEN * e + 4 * S)
        elif op == "rope":
            q = to_torch(normal(7, "op.q", (1, S, HEADS, HEAD_DIM), "bf16"), dev)
            k = to_torch(normal(7, "op.k", (1, S, HEADS, HEAD_DIM), "bf16"), dev)

            def fn():
                L.liger_rope_fwd(q, k, None, THETA)
                L.liger_rope_bwd(q, k, None, THETA)
            nbytes = 2 * (2 * 2 * S * HEADS * HEAD_DIM * e)
        else:
            g = to_torch(normal(7, "op.g", (S, INTER), "bf16"), dev)
            u = to_torch(normal(7, "op.u", (S, INTER), "bf16"), dev)
            dy = to_torch(normal(7, "op.sdy", (S, INTER), "bf16"), dev)
            y, dg, du = torch.empty_like(g), torch.empty_like(g), torch.empty_like(g)

            def fn():
                L.liger_swiglu_fwd(g, u, y)
                L.liger_swiglu_bwd(dy, g, u, dg, du)
            nbytes = 3 * S * INTER * e + 5 * S * INTER * e
        flops = None
    else:
        X = to_torch(normal(7, "op.mX", (S, HIDDEN), "bf16"), dev)
        Wg = to_torch(normal(7, "op.Wg", (INTER, HIDDEN), "bf16", 0.0, 0.02), dev)
        Wu = to_torch(normal(7, "op.Wu", (INTER, HIDDEN), "bf16", 0.0, 0.02), dev)
        out = torch.empty(S, INTER, dtype=bf, device=dev)
        if op == "fused_linear_swiglu":
            fn = lambda: L.liger_fused_linear_swiglu_fwd(X, Wg, Wu, out)
            flops = 4.0 * S * HIDDEN * INTER
        elif op == "fused_linear_swiglu_fwd_save":
            g, u = torch.empty_like(out), torch.empty_like(out)
            fn = lambda: L.liger_fused_linear_swiglu_fwd_save(X, Wg, Wu, out, g, u)
            flops = 4.0 * S * HIDDEN * INTER
        else:
            # the backward from the g, u of the saving forward: dG, dU, then dX and dW_g, dW_u
            g, u = torch.empty_like(out), torch.empty_like(out)
            L.liger_fused_linear_swiglu_fwd_save(X, Wg, Wu, out, g, u)
            dH = to_torch(normal(7, "op.mdH", (S, INTER), "bf16"), dev)
            dX, dWg, dWu = torch.empty_like(X), torch.empty_like(Wg), torch.empty_like(Wu)
            ws = torch.empty(L.liger_fused_linear_swiglu_workspace(S, INTER), dtype=torch.uint8, device=dev)
            fn = lambda: L.liger_fused_linear_swiglu_bwd_saved(X, Wg, Wu, dH, g, u, dX, dWg, dWu, ws)
            flops = 8.0 * S * HIDDEN * INTER
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / max(1, args.steps)
    rate = {"tflops": flops / ms / 1e9} if flops else {"gbs": nbytes / ms / 1e6}
    emit(dict({"op": op, "seq": S, "ms_per_call": ms, "steps": args.steps, "warmup": args.warmup,
               "note": "single operator alone (profiling case), not the benchmark step"}, **rate))
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return reference_arm(args)
    if args.op != "chain":
        return single_op(args)
    return native_arm(args)


if __name__ == "__main__":
    sys.exit(main())
