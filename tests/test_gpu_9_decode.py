"""GPU: the single-launch decode kernel (kt_mxfp4_moe_decode).

One cooperative launch runs routing, permutation, MXFP8 quantisation, FC1 +
SwiGLU, FC2 and the combine.  It must reproduce the multi-launch path
(kt_moe_route_permute then kt_mxfp4_moe_forward) bit for bit -- routing ids
and weights, expert offsets, permutation, A1, A2 and the bf16 output -- and
match the fp64 oracle (ids exact, output within 2e-2 normwise per token) at
the token counts 1/2/8/32 and on expert hit patterns with a never-picked
expert ("Kimi-K3 SM120 FlashInfer MXFP4 MoE", later hard gates, item 5), on
the tiny layer, on ragged shapes, on the Kimi-K3-shaped layer at T=16 and
under CUDA-graph replay.
"""
import numpy as np
import pytest
import torch

import mxfp4_weight_moe_gb300 as kt
import oracle as O
from mxfp4_weight_moe_gb300 import synthetic as syn

from helpers import OUT_RTOL, bf16_bits_np, bf16_to_f64, normwise_rel, oracle_subset, sample_tokens, ws_view

pytestmark = pytest.mark.gpu


def _inputs(T, H, E, k, I, recipe, seed=0):
    hidden = syn.make_hidden(T, H, seed, device="cuda")
    logits = syn.make_logits(T, E, recipe, seed, device="cuda")
    W = syn.make_weights(E, H, I, seed=seed, device="cuda")
    return hidden, logits, W


def _compare(hidden, logits, W, k, renormalize=True, opts=None, oracle_tokens=None):
    opts = opts or {}
    T, H = hidden.shape
    E, I2, _ = W[0].shape
    I = I2 // 2
    ws_d = torch.empty(kt.workspace_bytes(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    out_d, ids_d, w_d = kt.decode(logits, hidden, k, *W, renormalize=renormalize, workspace=ws_d, **opts)
    ws_f = torch.empty_like(ws_d)
    ids_f, w_f, *_ = kt.route_permute(logits, k, renormalize=renormalize)
    out_f = kt.forward(hidden, ids_f, w_f, *W, workspace=ws_f, **opts)
    torch.cuda.synchronize()
    assert kt.read_device_error(ws_d) == 0
    assert torch.equal(ids_d, ids_f) and torch.equal(w_d, w_f)
    lay = kt.workspace_layout(T, H, I, E, k)
    S = T * k
    for name, nbytes in (("expert_offsets", 4 * (E + 1)), ("perm", 4 * S), ("inv_perm", 4 * S), ("a1", S * H),
                         ("a2", S * I)):
        np.testing.assert_array_equal(ws_view(ws_d, lay[name], nbytes), ws_view(ws_f, lay[name], nbytes),
                                      err_msg=name)
    assert torch.equal(out_d.view(torch.int16), out_f.view(torch.int16))
    # against the oracle
    ids_np, w_np = O.route(logits.cpu().numpy(), k, renormalize=renormalize)
    np.testing.assert_array_equal(ids_d.cpu().numpy(), ids_np)
    assert np.abs(w_d.cpu().numpy() - w_np).max() <= 2 * np.spacing(np.float32(1.0))
    tokens = np.arange(T, dtype=np.int32) if oracle_tokens is None else oracle_tokens
    ref = oracle_subset(bf16_bits_np(hidden), ids_np, w_np, *W, tokens=tokens, want=("out_f64",), **opts)
    rel = normwise_rel(bf16_to_f64(bf16_bits_np(out_d)[tokens]), ref["out_f64"])
    assert rel.max() <= OUT_RTOL, rel.max()
    return out_d


@pytest.mark.parametrize("name", ["tiny", "small_T1", "small_T2", "small_T8", "small_T32"])
def test_decode_small_configs(name):
    cfg = syn.CONFIGS[name]
    hidden, logits, W = _inputs(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.logits, cfg.seed)
    _compare(hidden, logits, W, cfg.k)


@pytest.mark.parametrize("shape", [
    (25, 384, 2, 2, 640, "normal"),      # ragged K (3 and 5 quads), 25 rows per expert
    (7, 256, 5, 3, 128, "normal"),
    (24, 512, 3, 3, 256, "normal"),      # k = E
    (64, 1024, 32, 32, 512, "uniform"),  # 2048 slots: the decode kernel's largest batch
    (3, 1024, 1024, 8, 256, "normal"),   # E = 1024: most experts idle
    # above 4 tokens (or 16384 logits) routing runs as a warp per token across the grid and the
    # permutation in CTA 0, with grid barriers between; smaller batches route and permute in every CTA
    (64, 256, 512, 8, 128, "normal"),
    (4, 256, 1024, 8, 128, "normal"),     # 4 tokens over 1024 experts: in every CTA
    (128, 512, 256, 16, 256, "uniform"),  # 2048 slots on that path
])
def test_decode_ragged_shapes(shape):
    T, H, E, k, I, recipe = shape
    hidden, logits, W = _inputs(T, H, E, k, I, recipe, seed=3)
    _compare(hidden, logits, W, k)


def test_decode_full_softmax_and_variants():
    hidden, logits, W = _inputs(32, 1024, 16, 4, 512, "hot_cold", seed=4)
    _compare(hidden, logits, W, 4, renormalize=False)
    _compare(hidden, logits, W, 4, opts=dict(gate_up="interleaved", activation="swiglu_clamped", limit=0.5))


@pytest.mark.slow
def test_decode_kimi_shaped_t16():
    cfg = syn.CONFIGS["kimi_T16"]
    hidden, logits, W = _inputs(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.logits, cfg.seed)
    _compare(hidden, logits, W, cfg.k, oracle_tokens=np.array([0, 7, 15], np.int32))
    del W
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["small_T1", "small_T32"])
def test_decode_replays_in_cuda_graph(name):
    cfg = syn.CONFIGS[name]
    hidden, logits, W = _inputs(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.logits, cfg.seed)
    ws = torch.empty(kt.workspace_bytes(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k), dtype=torch.uint8, device="cuda")
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    topk = (torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda"),
            torch.empty(cfg.T, cfg.k, dtype=torch.float32, device="cuda"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        kt.decode(logits, hidden, cfg.k, *W, out=out, topk=topk, workspace=ws, stream=s)   # set-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kt.decode(logits, hidden, cfg.k, *W, out=out, topk=topk, workspace=ws, stream=s)
    hidden.copy_(syn.make_hidden(cfg.T, cfg.H, cfg.seed + 5, device="cuda"))
    logits.copy_(syn.make_logits(cfg.T, cfg.E, cfg.logits, cfg.seed + 5, device="cuda"))
    g.replay()
    torch.cuda.synchronize()
    assert kt.read_device_error(ws) == 0
    ids_np, w_np = O.route(logits.cpu().numpy(), cfg.k)
    np.testing.assert_array_equal(topk[0].cpu().numpy(), ids_np)
    ref = O.moe_forward(bf16_bits_np(hidden), ids_np, w_np, *[t.cpu().numpy() for t in W], want=("out_f64",))
    rel = normwise_rel(bf16_to_f64(bf16_bits_np(out)), ref["out_f64"])
    assert rel.max() <= OUT_RTOL, rel.max()


def test_decode_rejects_batches_above_its_limit():
    hidden, logits, W = _inputs(65, 128, 32, 32, 128, "normal")
    with pytest.raises(kt.KTError) as ei:
        kt.decode(logits, hidden, 32, *W)
    assert ei.value.status == -2


def test_decode_bounded_wait_expiry_is_reported():
    # each GEMM producer withholds its first stage: the MMA waits run out (0.1 s), the grid barriers after
    # them are bounded too, the kernel returns, and the context still works
    cfg = syn.CONFIGS["small_T8"]
    hidden, logits, W = _inputs(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.logits, cfg.seed)
    ws = torch.empty(kt.workspace_bytes(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k), dtype=torch.uint8, device="cuda")
    kt.debug_configure(100_000, kt.KT_DEBUG_WITHHOLD_STAGE)
    try:
        kt.decode(logits, hidden, cfg.k, *W, workspace=ws)
        torch.cuda.synchronize()
    finally:
        kt.debug_configure()
    code = kt.read_device_error(ws)
    assert code & (kt.KT_DEVERR_TIMEOUT_LOAD | kt.KT_DEVERR_TIMEOUT_MMA | kt.KT_DEVERR_TIMEOUT_EPI | 0x10)
    _compare(hidden, logits, W, cfg.k)
