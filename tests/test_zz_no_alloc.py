"""liger_rmsnorm_bwd_noalloc: the RMSNorm backward for callers that cannot
allocate device memory when they call it (an operator interface with no
workspace slot, a loop that must not call cudaMalloc because it can stall
the whole device, a process whose memory is all reserved at start-up).

It is called here through the C-ABI with raw device pointers, twice in a
row, and its dx / dw must match the workspace entry point's within the
tolerance the parity tests use.  This file is collected last so that a run
stopping at the first failure has already run every other test; it also
passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest

import datagen
import oracle
from gpu_util import TOL, dev, host

pytestmark = pytest.mark.gpu


def _case(lib, dtype, rows, cols):
    import torch
    x = datagen.normal(31, "nx", (rows, cols), dtype)
    w = datagen.normal(31, "nw", (cols,), dtype, 1.0, 0.1)
    dy = datagen.normal(31, "ndy", (rows, cols), dtype)
    tx, tw, tdy = dev(x), dev(w), dev(dy)
    y = torch.empty_like(tx)
    rstd = torch.empty(rows, dtype=torch.float32, device="cuda")
    lib.liger_rmsnorm_fwd(tx, tw, y, rstd, 1e-6)
    # reference: the entry point that takes a caller-provided workspace
    ws = torch.empty(lib.liger_rmsnorm_bwd_workspace(rows, cols), dtype=torch.uint8, device="cuda")
    dx_ref, dw_ref = torch.empty_like(tx), torch.empty_like(tw)
    lib.liger_rmsnorm_bwd(tdy, tx, tw, rstd, dx_ref, dw_ref, ws)
    raw = lib.load()
    code = lib.LIGER_F32 if dtype == "f32" else lib.LIGER_BF16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    odx, odw = oracle.rmsnorm_bwd(dy, x, w, 1e-6)
    for _ in range(2):                      # two calls in a row share the built-in scratch
        dx, dw = torch.full_like(tx, 7.0), torch.full_like(tw, 7.0)
        rc = raw.liger_rmsnorm_bwd_noalloc(tdy.data_ptr(), tx.data_ptr(), tw.data_ptr(), rstd.data_ptr(),
                                           dx.data_ptr(), dw.data_ptr(), rows, cols, code, stream)
        assert rc == 0, raw.liger_last_error().decode()
        torch.cuda.synchronize()
        assert oracle.rel_err(host(dx), host(dx_ref)) <= TOL[dtype]
        assert oracle.rel_err(host(dw), host(dw_ref)) <= TOL[dtype]
        # and against the fp64 oracle directly (the backward from the same stored inputs and
        # the forward's eps; the kernel reads the rstd the GPU forward wrote)
        assert oracle.rel_err(host(dx), odx) <= TOL[dtype]
        assert oracle.rel_err(host(dw), odw) <= TOL[dtype]
    return host(dw), host(dw_ref)


# the last two cases are wide enough that the scratch array bounds the number of
# partial rows: 16 MiB / (4 * 65536) = 64 partial rows for 2048 rows (bf16), and
# 16 MiB / (4 * 1048576) = 4 partial rows for 64 rows (fp32)
@pytest.mark.parametrize("dtype,rows,cols", [("bf16", 3000, 4096), ("f32", 257, 1000), ("bf16", 2048, 8192),
                                             ("bf16", 7, 33), ("bf16", 2048, 65536), ("f32", 64, 1048576)])
def test_noalloc_matches_workspace_entry_point(cuda_lib, dtype, rows, cols):
    _case(cuda_lib, dtype, rows, cols)


def test_noalloc_rejects_columns_beyond_its_scratch(cuda_lib):
    raw = cuda_lib.load()
    ok = ctypes.c_void_p(0x1000)             # never dereferenced: the size check comes first
    too_wide = (16 * 1024 * 1024) // 4 + 8
    rc = raw.liger_rmsnorm_bwd_noalloc(ok, ok, ok, ok, ok, ok, 4, too_wide, cuda_lib.LIGER_BF16, None)
    assert rc == -6
    assert "scratch" in raw.liger_last_error().decode()
