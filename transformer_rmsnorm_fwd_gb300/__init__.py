"""Fused decoder-layer operators for one NVIDIA GB300 GPU (sm_103a).

RMSNorm forward/backward, in-place RoPE on Q and K, the SwiGLU activation, a
fused linear cross-entropy that never materialises the [T x V] logits (token-
chunked, and a two-pass vocabulary-chunked variant),
FusedLinearSwiGLU (gate/up projections with the activation in the GEMM
epilogue) and the fused RMSNorm + QKV projection + RoPE forward, all
hand-written CUDA behind the C-ABI of ``libliger.so`` (``include/liger.h``).
This package is the Python binding of that library: see ``_native`` for the
functions, which carry the C entry points' names.
"""
from ._native import (LIGER_BF16, LIGER_F32, LigerError,  # noqa: F401
                      liger_device_status, liger_device_status_mark, liger_fused_linear_swiglu_bwd,
                      liger_fused_linear_swiglu_bwd_saved, liger_fused_linear_swiglu_fwd,
                      liger_fused_linear_swiglu_fwd_save,
                      liger_fused_linear_swiglu_workspace, liger_linear_ce_fwd_bwd, liger_linear_ce_two_pass_fwd_bwd,
                      liger_linear_ce_two_pass_workspace, liger_linear_ce_workspace,
                      liger_rmsnorm_bwd, liger_rmsnorm_bwd_noalloc, liger_rmsnorm_bwd_workspace, liger_rmsnorm_fwd,
                      liger_rmsnorm_qkv_rope_fwd, liger_rmsnorm_qkv_rope_workspace, liger_rope_bwd,
                      liger_rope_bwd_ex, liger_rope_fwd, liger_rope_fwd_ex, liger_swiglu_bwd, liger_swiglu_fwd, load)
