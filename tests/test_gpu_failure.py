"""Failure detection on the GPU without a fault: the bounded look-back wait
runs out on purpose (a predecessor that never publishes), the kernel flags
the error and returns, the host reads GS_ERR_TIMEOUT, and the context keeps
working afterwards.  Capacity overflow and argument errors are checked in
test_gpu_parity.py and test_abi_cpu.py."""
import numpy as np
import pytest
import torch

import scenes
from parity_util import f32_cams

pytestmark = pytest.mark.gpu


def test_lookback_wait_times_out_and_context_survives():
    import __graft_entry__
    __graft_entry__.build()
    import gaussian_splatting_differentiable_gs_gb300 as gs
    L = gs.lib()
    L.gs_selftest_lookback_timeout.restype = int
    import ctypes as C
    L.gs_selftest_lookback_timeout.argtypes = [C.c_void_p, C.c_size_t, C.c_void_p]
    ws = torch.zeros(gs.gs_bin_workspace_bytes(1, 1), dtype=torch.uint8, device="cuda")
    st = L.gs_selftest_lookback_timeout(ws.data_ptr(), ws.numel(),
                                        torch.cuda.current_stream().cuda_stream)
    assert st == gs.GS_ERR_TIMEOUT
    # the status word was read and cleared; the context still runs a full step
    assert gs.gs_workspace_status(ws) == gs.GS_OK
    cfg = scenes.make("tiny_2k_256", n_override=300)
    step = gs.TrainStep(torch.from_numpy(cfg["params"]).cuda(), f32_cams(cfg["cams"]),
                        torch.from_numpy(cfg["target"]).cuda())
    step.step()
    torch.cuda.synchronize()
    assert np.isfinite(step.loss.item())
