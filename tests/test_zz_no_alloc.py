"""The allocation-free routing entry point (kt_moe_route_permute_noalloc).

Some callers cannot allocate device memory -- a plugin whose host framework
owns all GPU memory and hands it no workspace, or a serving loop that must
not pay cudaMalloc's implicit synchronisation -- so the library offers one
variant of route + permute whose scratch is a fixed device array inside the
library.  Its outputs must equal kt_moe_route_permute's (workspace version)
exactly, on consecutive calls that reuse that shared array.  This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import mxfp4_weight_moe_gb300 as kt
from mxfp4_weight_moe_gb300 import synthetic as syn


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # checked before anything touches the GPU: T=65536, E=1024, k=32 needs far more than 1 MiB
    P = ctypes.c_void_p(0x7F0000000000)
    need = int(kt.lib().kt_moe_route_workspace_bytes(65536, 1024, 32))
    assert need > kt.KT_NOALLOC_SCRATCH_BYTES
    st = kt.lib().kt_moe_route_permute_noalloc(P, 65536, 1024, 32, 1, P, P, P, P, P, None)
    assert st == -3                                     # KT_ERR_WORKSPACE
    assert "static scratch" in kt.lib().kt_last_error().decode()


def test_noalloc_checks_arguments_before_the_size_limit():
    # the same order of checks as the workspace entry point: a null or misaligned pointer is reported as
    # such even when the sizes are also beyond the static scratch
    P = ctypes.c_void_p(0x7F0000000000)
    st = kt.lib().kt_moe_route_permute_noalloc(None, 65536, 1024, 32, 1, P, P, P, P, P, None)
    assert st == -1                                     # KT_ERR_INVALID_ARG
    Q = ctypes.c_void_p(0x7F0000000002)
    st = kt.lib().kt_moe_route_permute_noalloc(P, 65536, 1024, 32, 1, Q, P, P, P, P, None)
    assert st == -7                                     # KT_ERR_ALIGNMENT
    st = kt.lib().kt_moe_route_permute_noalloc(P, 8, 16, 17, 1, P, P, P, P, P, None)
    assert st == -1                                     # k > E
    assert kt.lib().kt_moe_route_permute_noalloc(P, 0, 16, 4, 1, P, P, P, P, P, None) == 0   # T = 0: no-op


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["small_T32", "kimi_T8192"])
def test_noalloc_matches_workspace_entry_on_consecutive_calls(name):
    cfg = syn.CONFIGS[name]
    assert int(kt.lib().kt_moe_route_workspace_bytes(cfg.T, cfg.E, cfg.k)) <= kt.KT_NOALLOC_SCRATCH_BYTES
    for call in range(3):
        logits = syn.make_logits(cfg.T, cfg.E, cfg.logits, seed=cfg.seed + call, device="cuda")
        ref = kt.route_permute(logits, cfg.k)
        outs = tuple(torch.empty_like(r) for r in ref)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        got = kt.route_permute_noalloc(logits, cfg.k, out=outs)
        torch.cuda.synchronize()
        if call >= 1:
            # the call itself takes no device memory (the first call may load the module's code)
            assert torch.cuda.mem_get_info()[0] == free0, f"call {call}: device memory changed"
        for g, r, what in zip(got, ref, ("topk_ids", "topk_w", "expert_offsets", "perm", "inv_perm")):
            assert torch.equal(g, r), f"call {call}: {what} differs from the workspace entry point"
        assert int(got[2][-1]) == cfg.T * cfg.k
