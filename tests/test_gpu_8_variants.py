"""GPU: the gated-FC1 options (interleaved gate/up rows, clamped SwiGLU)
against the fp64 oracle run with the same options.

"Kimi-K3 SM120 FlashInfer MXFP4 MoE" (Phase 0 audit conclusions, item 4)
names the GPT-OSS SwiGLU weight layout and parameters; they are read as the
published GPT-OSS definition (row 2i gate i, row 2i+1 up i; h = min(g, L) *
sigmoid(alpha * min(g, L)) * (clamp(u, -L, L) + 1)).  Checked: A1 bit-exact,
A2 within one code step on <= 0.1 % of elements, bf16 output within 2e-2
normwise per token; a limit small enough to clamp most values exercises the
clamp.  The interleaved layout must also reproduce, bit for bit, the halves
layout run on the same rows reordered.
"""
import numpy as np
import pytest
import torch

import mxfp4_weight_moe_gb300 as kt
import oracle as O
from mxfp4_weight_moe_gb300 import synthetic as syn

from helpers import OUT_RTOL, bf16_bits_np, bf16_to_f64, check_a2, normwise_rel, oracle_subset, sample_tokens, \
    scale_flips_valid, ws_view

pytestmark = pytest.mark.gpu


def _case(T, H, E, k, I, recipe, seed, sf_boost=0):
    hidden = syn.make_hidden(T, H, seed, device="cuda")
    ids, w = O.route(syn.make_logits(T, E, recipe, seed, device="cpu").numpy(), k)
    W = list(syn.make_weights(E, H, I, seed=seed, device="cuda"))
    if sf_boost:
        W[1] = (W[1].int() + sf_boost).to(torch.uint8)    # larger gate / up values, so a limit bites
    return hidden, ids, w, W


def _check(hidden, ids_np, w_np, W, tokens, **opts):
    T, H = hidden.shape
    k = ids_np.shape[1]
    E, I2, _ = W[0].shape
    I = I2 // 2
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np).cuda()
    ws = torch.empty(kt.workspace_bytes(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    out = kt.forward(hidden, ids, w, *W, workspace=ws, **opts)
    torch.cuda.synchronize()
    assert kt.read_device_error(ws) == 0
    lay = kt.workspace_layout(T, H, I, E, k)
    S = T * k
    hbits = bf16_bits_np(hidden)
    ref = oracle_subset(hbits, ids_np, w_np, *W, tokens=tokens, want=("out_f64", "a2", "a2_sf"), **opts)
    _, _, rinv, _ = O.permute(ids_np, E)
    a2 = ws_view(ws, lay["a2"], S * I).reshape(S, I)
    a2_sf = kt.scales_from_kstep_major(ws[lay["a2_sf"]:], S, I).cpu().numpy()
    gc, gs, rc, rs = [], [], [], []
    for i, t in enumerate(tokens):
        for j in range(k):
            p = rinv[t * k + j]
            gc.append(a2[p]); gs.append(a2_sf[p]); rc.append(ref["a2"][i, j]); rs.append(ref["a2_sf"][i, j])
    frac, worst = check_a2(np.array(gc), np.array(gs), np.array(rc), np.array(rs))
    assert frac <= 1e-3 and worst <= 1.0 + 1e-9, (frac, worst)
    n_sf, bad_sf = scale_flips_valid(np.array(gc), np.array(gs), np.array(rc), np.array(rs))
    assert bad_sf == 0, (n_sf, bad_sf)
    rel = normwise_rel(bf16_to_f64(bf16_bits_np(out)[tokens]), ref["out_f64"])
    assert rel.max() <= OUT_RTOL, rel.max()
    return out


@pytest.mark.parametrize("gate_up,activation,limit", [
    ("interleaved", "swiglu", 7.0),
    ("halves", "swiglu_clamped", 0.25),
    ("interleaved", "swiglu_clamped", 0.25),
    ("interleaved", "swiglu_clamped", 7.0),
])
@pytest.mark.parametrize("shape", [
    (32, 1024, 16, 4, 512, "hot_cold"),     # small_T32: K % 512 == 0, scales by TMA
    (25, 384, 2, 2, 640, "normal"),         # ragged: K = 3 quads, scales by cp.async gathers
    (1, 128, 2, 2, 128, "normal"),          # the tiny layer
    (256, 512, 4, 2, 256, "normal"),        # 128 rows per expert: prefill-sized tiles in 2-CTA clusters
])
def test_variant_against_oracle(gate_up, activation, limit, shape):
    T, H, E, k, I, recipe = shape
    hidden, ids, w, W = _case(T, H, E, k, I, recipe, seed=5, sf_boost=3)
    _check(hidden, ids, w, W, np.arange(T, dtype=np.int32), gate_up=gate_up, activation=activation, alpha=1.702,
           limit=limit)


@pytest.mark.parametrize("activation", ["swiglu", "swiglu_clamped"])
@pytest.mark.parametrize("shape", [(32, 1024, 16, 4, 512), (25, 384, 2, 2, 640)])
def test_interleaved_rows_reproduce_halves_layout(activation, shape):
    T, H, E, k, I = shape
    hidden, ids_np, w_np, W = _case(T, H, E, k, I, "normal", seed=6)
    order = torch.empty(2 * I, dtype=torch.long)
    order[0::2] = torch.arange(I)
    order[1::2] = I + torch.arange(I)
    order = order.cuda()
    W_int = [W[0].index_select(1, order).contiguous(), W[1].index_select(1, order).contiguous(), W[2], W[3]]
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np).cuda()
    a = kt.forward(hidden, ids, w, *W, gate_up="halves", activation=activation, limit=0.5)
    b = kt.forward(hidden, ids, w, *W_int, gate_up="interleaved", activation=activation, limit=0.5)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.slow
def test_variant_dsv4_shaped_sample():
    cfg = syn.CONFIGS["dsv4"]
    hidden, ids, w, W = _case(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.logits, cfg.seed)
    tokens = sample_tokens(ids, 64, seed=3)
    _check(hidden, ids, w, W, tokens, gate_up="interleaved", activation="swiglu_clamped", alpha=1.702, limit=7.0)


def test_options_are_checked():
    hidden, ids_np, w_np, W = _case(1, 128, 2, 2, 128, "normal", seed=1)
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np).cuda()
    for bad in (dict(activation="swiglu_clamped", limit=0.0), dict(activation="swiglu_clamped", limit=float("inf")),
                dict(activation="swiglu_clamped", alpha=float("nan"))):
        with pytest.raises(kt.KTError):
            kt.forward(hidden, ids, w, *W, **bad)
    with pytest.raises(ValueError):
        kt.forward(hidden, ids, w, *W, gate_up="rows")
