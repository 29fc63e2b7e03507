"""Every entry point except the two linear cross-entropies (which wait on the
host for their label scan) queues work only, so after a first eager call it
can be captured in a CUDA graph: RMSNorm fwd/bwd, RoPE fwd/bwd, SwiGLU
fwd/bwd, FusedLinearSwiGLU fwd/bwd, the fused RMSNorm + QKV + RoPE and the
no-allocation RMSNorm backward, captured into one graph and replayed; the
kernels are deterministic, so the replay reproduces the eager results bit for
bit."""
import pytest

pytestmark = pytest.mark.gpu


def test_capture_and_replay_matches_eager(cuda_lib):
    import torch
    L = cuda_lib
    torch.manual_seed(3)
    dev = "cuda"
    T, H, I, Hq, D = 512, 256, 512, 2, 64
    bf = torch.bfloat16
    x = torch.randn(T, H, device=dev).to(bf)
    w = (1 + 0.1 * torch.randn(H, device=dev)).to(bf)
    dy = torch.randn(T, H, device=dev).to(bf)
    q0 = torch.randn(1, T, Hq, D, device=dev).to(bf)
    k0 = torch.randn(1, T, Hq, D, device=dev).to(bf)
    g = torch.randn(T, I, device=dev).to(bf)
    u = torch.randn(T, I, device=dev).to(bf)
    dh = torch.randn(T, I, device=dev).to(bf)
    Wg = (0.05 * torch.randn(I, H, device=dev)).to(bf)
    Wu = (0.05 * torch.randn(I, H, device=dev)).to(bf)
    Wq = (0.05 * torch.randn(Hq * D, H, device=dev)).to(bf)
    outs = {
        "y": torch.empty_like(x), "rstd": torch.empty(T, device=dev), "dx": torch.empty_like(x),
        "dw": torch.empty_like(w), "dx2": torch.empty_like(x), "dw2": torch.empty_like(w),
        "q": torch.empty_like(q0), "k": torch.empty_like(k0), "h": torch.empty_like(g), "dg": torch.empty_like(g),
        "du": torch.empty_like(g), "lh": torch.empty(T, I, device=dev, dtype=bf), "ldX": torch.empty_like(x),
        "ldWg": torch.empty_like(Wg), "ldWu": torch.empty_like(Wu), "qq": torch.empty(1, T, Hq, D, device=dev, dtype=bf),
        "qk": torch.empty(1, T, Hq, D, device=dev, dtype=bf), "qv": torch.empty(1, T, Hq, D, device=dev, dtype=bf),
    }
    ws_r = torch.empty(L.liger_rmsnorm_bwd_workspace(T, H), dtype=torch.uint8, device=dev)
    ws_s = torch.empty(L.liger_fused_linear_swiglu_workspace(T, I), dtype=torch.uint8, device=dev)
    ws_q = torch.empty(L.liger_rmsnorm_qkv_rope_workspace(T, H, Hq, Hq, D), dtype=torch.uint8, device=dev)

    def step(o):
        L.liger_rmsnorm_fwd(x, w, o["y"], o["rstd"], 1e-6)
        L.liger_rmsnorm_bwd(dy, x, w, o["rstd"], o["dx"], o["dw"], ws_r)
        L.liger_rmsnorm_bwd_noalloc(dy, x, w, o["rstd"], o["dx2"], o["dw2"])
        o["q"].copy_(q0)
        o["k"].copy_(k0)
        L.liger_rope_fwd(o["q"], o["k"], None, 1e4)
        L.liger_rope_bwd(o["q"], o["k"], None, 1e4)
        L.liger_rope_fwd(o["q"], o["k"], None, 1e4)
        L.liger_swiglu_fwd(g, u, o["h"])
        L.liger_swiglu_bwd(dh, g, u, o["dg"], o["du"])
        L.liger_fused_linear_swiglu_fwd(x, Wg, Wu, o["lh"])
        L.liger_fused_linear_swiglu_bwd(x, Wg, Wu, dh, o["ldX"], o["ldWg"], o["ldWu"], ws_s)
        L.liger_rmsnorm_qkv_rope_fwd(x, w, Wq, Wq, Wq, o["qq"], o["qk"], o["qv"], ws_q, 1, T, Hq, Hq, D)

    # eager: the first calls set up the library's per-device state; the second are the reference
    step(outs)
    eager = {k: torch.empty_like(v) for k, v in outs.items()}
    step(eager)
    torch.cuda.synchronize()
    for v in outs.values():
        v.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step(outs)
    torch.cuda.current_stream().wait_stream(s)
    graph.replay()
    torch.cuda.synchronize()
    for k in outs:
        a, b = outs[k], eager[k]
        if a.dtype == bf:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), k
