"""liger_device_status: the read-back of the library-owned words in which the
staged RMSNorm and RoPE kernels, FusedLinearSwiGLU and the fused RMSNorm +
QKV + RoPE record an expired bounded wait.  Normal calls leave every word clear; a word
marked by the test hook (nothing expires, no GPU fault) is reported as
LIGER_ERR_CUDA naming its family, and is clear again after the read."""
import pytest

import datagen
from gpu_util import dev

pytestmark = pytest.mark.gpu


def test_clear_after_normal_calls(cuda_lib):
    import torch
    x = dev(datagen.normal(51, "dsx", (300, 4096), "bf16"))
    w = dev(datagen.normal(51, "dsw", (4096,), "bf16", 1.0, 0.1))
    y, rstd = torch.empty_like(x), torch.empty(300, dtype=torch.float32, device="cuda")
    cuda_lib.liger_rmsnorm_fwd(x, w, y, rstd, 1e-6)
    ws = torch.empty(cuda_lib.liger_rmsnorm_bwd_workspace(300, 4096), dtype=torch.uint8, device="cuda")
    dx, dw = torch.empty_like(x), torch.empty_like(w)
    cuda_lib.liger_rmsnorm_bwd(y, x, w, rstd, dx, dw, ws)
    Wg = dev(datagen.normal(51, "dsg", (512, 4096), "bf16", 0.0, 0.02))
    out = torch.empty(300, 512, dtype=torch.bfloat16, device="cuda")
    cuda_lib.liger_fused_linear_swiglu_fwd(x, Wg, Wg, out)
    qk = dev(datagen.normal(51, "dsq", (1, 300, 4, 128), "bf16"))
    cuda_lib.liger_rope_fwd(qk, None, None, 1e4)
    cuda_lib.liger_device_status()          # raises if any word is set


@pytest.mark.parametrize("which,name", [(0, "RMSNorm"), (1, "FusedLinearSwiGLU"), (2, "QKV"), (3, "RoPE")])
def test_marked_word_is_reported_once(cuda_lib, which, name):
    cuda_lib.liger_device_status()
    cuda_lib.liger_device_status_mark(which)
    with pytest.raises(cuda_lib.LigerError) as e:
        cuda_lib.liger_device_status()
    assert e.value.status == -7 and name in str(e.value)
    cuda_lib.liger_device_status()          # read and cleared
