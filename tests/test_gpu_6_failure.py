"""GPU: the device-side failure path, without faulting or hanging the GPU.

A test hook shortens every GEMM barrier wait to 0.1 s and makes each CTA's
producer withhold one pipeline stage (nothing is loaded into it and it is
never signalled), so the MMA issuer's wait runs out.  The kernel must record
a timeout in the device error word, free its tensor memory and return; the
host reads KT_ERR_DEVICE_TIMEOUT and the same process then runs a normal
forward that still matches the oracle.
"""
import pytest
import torch

import mxfp4_weight_moe_gb300 as kt

from test_gpu_3_forward import _check_case, _inputs

pytestmark = pytest.mark.gpu


def test_gemm_wait_timeout_is_reported_and_context_survives():
    hidden, ids, w, W = _inputs(T=64, H=512, E=4, k=2, I=256, seed=21)
    T, H = hidden.shape
    ws = torch.empty(kt.workspace_bytes(T, H, 256, 4, 2), dtype=torch.uint8, device="cuda")
    ids_t, w_t = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    kt.debug_configure(wait_limit_us=100_000, flags=kt.KT_DEBUG_WITHHOLD_STAGE)
    try:
        kt.forward(hidden, ids_t, w_t, *W, workspace=ws)
        code = kt.read_device_error(ws)
    finally:
        kt.debug_configure()
    assert code & kt.KT_DEVERR_TIMEOUT_MMA, hex(code)
    # the context is still usable and results are correct afterwards
    _check_case(hidden, ids, w, W)
