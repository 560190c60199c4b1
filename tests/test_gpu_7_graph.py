"""GPU: routing + the layer forward captured in a CUDA graph and replayed.

The forward enqueues only stream-ordered work (a memset and kernel launches
whose tensor maps are encoded on the host at enqueue time), so with
preallocated outputs and workspaces the whole step captures into one graph.
Replays must give bit-identical results to eager calls, including after the
inputs are overwritten in place, and the replayed output must match the fp64
oracle on those new inputs (token counts 1 and 32 and the DeepSeek-V4-Flash-
shaped prefill: "Kimi-K3 SM120 FlashInfer MXFP4 MoE", later hard gates,
item 5, asks for CUDA Graph capture/replay coverage at such token counts).
"""
import numpy as np
import pytest
import torch

import mxfp4_weight_moe_gb300 as kt
import oracle as O
from mxfp4_weight_moe_gb300 import synthetic as syn

from helpers import OUT_RTOL, bf16_bits_np, bf16_to_f64, normwise_rel, oracle_subset, sample_tokens

pytestmark = pytest.mark.gpu


def _setup(name):
    cfg = syn.CONFIGS[name]
    dev = torch.device("cuda")
    T, H, E, k, I = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
    hidden = syn.make_hidden(T, H, cfg.seed, device=dev)
    logits = syn.make_logits(T, E, cfg.logits, cfg.seed, device=dev)
    W = syn.make_weights(E, H, I, seed=cfg.seed, device=dev)
    route_out = (torch.empty(T, k, dtype=torch.int32, device=dev), torch.empty(T, k, dtype=torch.float32, device=dev),
                 torch.empty(E + 1, dtype=torch.int32, device=dev), torch.empty(T * k, dtype=torch.int32, device=dev),
                 torch.empty(T * k, dtype=torch.int32, device=dev))
    ws_route = torch.empty(int(kt.lib().kt_moe_route_workspace_bytes(T, E, k)), dtype=torch.uint8, device=dev)
    ws = torch.empty(kt.workspace_bytes(T, H, I, E, k), dtype=torch.uint8, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)

    def step():
        ids, w, *_ = kt.route_permute(logits, k, out=route_out, workspace=ws_route)
        kt.forward(hidden, ids, w, *W, out=out, workspace=ws)

    return cfg, hidden, logits, out, ws, step, W


@pytest.mark.parametrize("name", ["small_T1", "small_T32", "dsv4"])
def test_step_replays_in_cuda_graph(name):
    cfg, hidden, logits, out, ws, step, W = _setup(name)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                      # first call on this device: launch attributes are set outside the capture
    torch.cuda.synchronize()
    ref = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert kt.read_device_error(ws) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # new inputs written in place: the replay must follow them exactly as an eager step does
    hidden.copy_(syn.make_hidden(cfg.T, cfg.H, cfg.seed + 1, device=hidden.device))
    logits.copy_(syn.make_logits(cfg.T, cfg.E, cfg.logits, cfg.seed + 1, device=logits.device))
    g.replay()
    torch.cuda.synchronize()
    got = out.clone()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), out.view(torch.int16))
    assert not torch.equal(got.view(torch.int16), ref.view(torch.int16))
    # the replayed output against the oracle on the new inputs
    ids, w = O.route(logits.cpu().numpy(), cfg.k)
    tokens = sample_tokens(ids, 64, seed=2)
    want = oracle_subset(bf16_bits_np(hidden), ids, w, *W, tokens=tokens, want=("out_f64",))["out_f64"]
    rel = normwise_rel(bf16_to_f64(bf16_bits_np(got)[tokens]), want)
    assert rel.max() <= OUT_RTOL, rel.max()
