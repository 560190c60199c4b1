"""GPU: the fused layer forward against the fp64 oracle.

Checked per call: the permutation in the workspace (bit-exact), the MXFP8
activations A1 (bit-exact: both sides quantise exact bf16 values with the
same rule), the requantised SwiGLU output A2 (codes may differ by one step
on <= 0.1 % of elements where fp32 and fp64 h straddle a rounding
boundary), and the bf16 output (normwise relative error per token <= 2e-2).
"""
import numpy as np
import pytest
import torch

import mxfp4_weight_moe_gb300 as kt
import oracle as O
from mxfp4_weight_moe_gb300 import synthetic as syn

from helpers import OUT_RTOL, bf16_bits_np, bf16_to_f64, check_a2, normwise_rel, oracle_subset, sample_tokens, \
    scale_flips_valid, \
    ws_view

pytestmark = pytest.mark.gpu


def _run_forward(hidden, ids, w, W):
    T, H = hidden.shape
    k = ids.shape[1]
    E, I2, _ = W[0].shape
    I = I2 // 2
    ws = torch.empty(kt.workspace_bytes(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    out = kt.forward(hidden, ids, w, *W, workspace=ws)
    torch.cuda.synchronize()
    return out, ws, kt.workspace_layout(T, H, I, E, k)


def _check_case(hidden, ids_np, w_np, W, tokens=None, check_a=True):
    """Run the GPU forward and compare with the oracle (on `tokens`, default all)."""
    T, H = hidden.shape
    k = ids_np.shape[1]
    E, I2, _ = W[0].shape
    I = I2 // 2
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np).cuda()
    out, ws, lay = _run_forward(hidden, ids, w, W)
    err = kt.read_device_error(ws)
    valid = (ids_np >= 0) & (ids_np < E)
    assert err == (0 if valid.all() else kt.KT_DEVERR_BAD_EXPERT_ID)
    hbits = bf16_bits_np(hidden)
    S = T * k
    # permutation (bit-exact)
    roff, rperm, rinv, bad = O.permute(ids_np, E)
    offs = ws_view(ws, lay["expert_offsets"], 4 * (E + 1)).view(np.int32)
    perm = ws_view(ws, lay["perm"], 4 * S).view(np.int32)
    inv = ws_view(ws, lay["inv_perm"], 4 * S).view(np.int32)
    np.testing.assert_array_equal(offs, roff)
    nvalid = int(roff[-1])
    np.testing.assert_array_equal(perm[:nvalid], rperm[:nvalid])
    np.testing.assert_array_equal(inv, rinv)
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    # A1 (bit-exact) on the rows of the checked tokens
    if check_a:
        a1 = ws_view(ws, lay["a1"], S * H).reshape(S, H)
        a1_sf = kt.scales_from_kstep_major(ws[lay["a1_sf"]:], S, H).cpu().numpy()
        rc, rs = O.quant_rows_bf16(hbits[tokens])
        for i, t in enumerate(tokens):
            for j in range(k):
                p = rinv[t * k + j]
                if p < 0:
                    continue
                np.testing.assert_array_equal(a1[p], rc[i], err_msg=f"A1 codes token {t} slot {j}")
                np.testing.assert_array_equal(a1_sf[p], rs[i], err_msg=f"A1 scales token {t} slot {j}")
    ref = oracle_subset(hbits, ids_np, w_np, *W, tokens=tokens, want=("out", "out_f64", "a2", "a2_sf"))
    # A2: codes at the permuted rows of the checked slots
    if check_a:
        a2 = ws_view(ws, lay["a2"], S * I).reshape(S, I)
        a2_sf = kt.scales_from_kstep_major(ws[lay["a2_sf"]:], S, I).cpu().numpy()
        gc, gs, rc2, rs2 = [], [], [], []
        for i, t in enumerate(tokens):
            for j in range(k):
                p = rinv[t * k + j]
                if p < 0:
                    continue
                gc.append(a2[p]); gs.append(a2_sf[p]); rc2.append(ref["a2"][i, j]); rs2.append(ref["a2_sf"][i, j])
        frac, worst = check_a2(np.array(gc), np.array(gs), np.array(rc2), np.array(rs2))
        assert frac <= 1e-3 and worst <= 1.0 + 1e-9, (frac, worst)
        n_sf, bad_sf = scale_flips_valid(np.array(gc), np.array(gs), np.array(rc2), np.array(rs2))
        assert bad_sf == 0, f"{bad_sf} of {n_sf} A2 scale differences are not a power-of-two straddle"
    got = bf16_to_f64(bf16_bits_np(out)[tokens])
    rel = normwise_rel(got, ref["out_f64"])
    assert rel.max() <= OUT_RTOL, f"max normwise rel err {rel.max():.3e} at token {tokens[int(rel.argmax())]}"
    return rel.max()


def _inputs(name=None, T=None, H=None, E=None, k=None, I=None, recipe="normal", seed=0):
    if name is not None:
        cfg = syn.CONFIGS[name]
        T, H, E, k, I, recipe, seed = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.logits, cfg.seed
    hidden = syn.make_hidden(T, H, seed, device="cuda")
    logits = syn.make_logits(T, E, recipe, seed, device="cpu")
    ids, w = O.route(logits.numpy(), k)
    W = syn.make_weights(E, H, I, seed=seed, device="cuda")
    return hidden, ids, w, W


@pytest.mark.parametrize("name", ["tiny", "small_T1", "small_T2", "small_T8", "small_T32"])
def test_forward_small_configs(name):
    _check_case(*_inputs(name))


@pytest.mark.parametrize("shape", [
    (25, 384, 2, 2, 640),      # 25 rows per expert (32-row tiles with a lead), K = 3 and 5 quads, FC2 unclustered
    (7, 256, 5, 3, 128),       # K = 2 and 1 quads (a 256-K stage over a single quad)
    (24, 512, 3, 3, 256),      # k = E: every expert gets every token
])
def test_forward_decode_shapes(shape):
    """Decode-sized ragged layers (T <= 25)."""
    T, H, E, k, I = shape
    _check_case(*_inputs(T=T, H=H, E=E, k=k, I=I, seed=11))


@pytest.mark.parametrize("shape", [
    (37, 384, 5, 2, 384),      # ragged: 3 K steps, 6 FC1 feature tiles, 3 FC2 tiles
    (600, 256, 4, 1, 128),     # ~150 tokens per expert: token chunks, odd tails
    (300, 128, 3, 3, 256),     # k = E, every expert gets every token (2 chunks of 150)
    (129, 256, 8, 2, 512),
    # prefill-sized: ~267 rows per expert in two chunks, one-quad stages in 2-CTA clusters
    (400, 384, 3, 2, 640),     # FC1 with K = 3 quads; FC2 (3 feature tiles) unclustered
    (400, 512, 3, 2, 640),     # FC2 clustered with K = 5 quads
])
def test_forward_ragged_shapes(shape):
    T, H, E, k, I = shape
    _check_case(*_inputs(T=T, H=H, E=E, k=k, I=I, seed=T))


def test_forward_all_tokens_one_expert():
    T, H, E, k, I = 700, 256, 4, 1, 256
    hidden, ids, w, W = _inputs(T=T, H=H, E=E, k=k, I=I, seed=5)
    ids[:] = 2                              # 700 rows on one expert: 3 chunks; three experts idle
    w[:] = 1.0
    _check_case(hidden, ids, w, W)


def test_forward_invalid_ids_skip_slot():
    hidden, ids, w, W = _inputs(T=64, H=256, E=6, k=3, I=256, seed=6)
    ids[3, 1] = 6
    ids[10, 0] = -1
    _check_case(hidden, ids, w, W)


def test_forward_zero_tokens():
    W = syn.make_weights(2, 128, 128, device="cuda")
    out = kt.forward(torch.empty(0, 128, dtype=torch.bfloat16, device="cuda"),
                     torch.empty(0, 2, dtype=torch.int32, device="cuda"),
                     torch.empty(0, 2, dtype=torch.float32, device="cuda"), *W)
    assert out.shape == (0, 128)


def test_forward_zero_weights_give_zero():
    hidden, ids, w, W = _inputs(T=20, H=128, E=2, k=2, I=128, seed=7)
    W = (torch.zeros_like(W[0]), W[1], W[2], W[3])
    out, ws, _ = _run_forward(hidden, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), W)
    assert torch.all(out.float() == 0)


def test_profile_records_only_the_selected_stages():
    hidden, ids, w, W = _inputs(T=32, H=512, E=4, k=2, I=256, seed=3)
    ids_t, w_t = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    kt.profile_enable(True, stages=("fc1",))
    try:
        kt.forward(hidden, ids_t, w_t, *W)
        kt.forward(hidden, ids_t, w_t, *W)
        prof = kt.profile_read()
    finally:
        kt.profile_enable(False)
    assert prof["fc1"][1] == 2 and prof["fc1"][0] > 0
    assert all(n == 0 for name, (_, n) in prof.items() if name != "fc1")


def test_forward_is_deterministic():
    hidden, ids, w, W = _inputs("small_T32")
    ids_t, w_t = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    a = kt.forward(hidden, ids_t, w_t, *W)
    b = kt.forward(hidden, ids_t, w_t, *W)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_forward_token_order_invariance():
    hidden, ids, w, W = _inputs(T=96, H=256, E=8, k=2, I=256, seed=8)
    p = np.random.default_rng(0).permutation(96)
    a = kt.forward(hidden, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), *W)
    b = kt.forward(hidden[torch.from_numpy(p).cuda()], torch.from_numpy(ids[p]).cuda(),
                   torch.from_numpy(w[p]).cuda(), *W)
    torch.cuda.synchronize()
    assert torch.equal(a[torch.from_numpy(p).cuda()].view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("shape,opts", [
    ((32, 1024, 16, 4, 512), {}),
    ((600, 256, 4, 1, 128), {}),
    ((400, 512, 3, 2, 640), {}),
    ((25, 384, 2, 2, 640), dict(gate_up="interleaved", activation="swiglu_clamped", limit=0.5)),
])
def test_forward_on_a_given_routing_matches_forward(shape, opts):
    """kt_mxfp4_moe_forward_routed reuses route_permute's permutation: bit-identical output, A1 and A2."""
    T, H, E, k, I = shape
    g = torch.Generator(device="cpu").manual_seed(T + H)
    hidden = syn.make_hidden(T, H, seed=T, device="cuda")
    logits = torch.randn(T, E, generator=g).cuda()
    W = syn.make_weights(E, H, I, seed=3, device="cuda")
    ids, w, offs, perm, inv = kt.route_permute(logits, k)
    ws_a = torch.empty(kt.workspace_bytes(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty_like(ws_a)
    out_a = kt.forward(hidden, ids, w, *W, workspace=ws_a, **opts)
    out_b = kt.forward(hidden, ids, w, *W, workspace=ws_b, routing=(offs, perm, inv), **opts)
    torch.cuda.synchronize()
    assert kt.read_device_error(ws_a) == 0 and kt.read_device_error(ws_b) == 0
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    lay = kt.workspace_layout(T, H, I, E, k)
    S = T * k
    for name, nbytes in (("a1", S * H), ("a2", S * I)):
        assert torch.equal(ws_a[lay[name]:lay[name] + nbytes], ws_b[lay[name]:lay[name] + nbytes]), name


@pytest.mark.parametrize("shape,opts,single", [
    ((32, 1024, 16, 4, 512), {}, True),                                 # decode-sized, one launch
    ((32, 1024, 16, 4, 512), {}, False),                                # decode-sized, routing + routed forward
    ((600, 256, 4, 1, 128), {}, False),
    ((25, 384, 2, 2, 640), dict(gate_up="interleaved", activation="swiglu_clamped", limit=0.5), True),
])
def test_moe_layer_matches_route_and_forward(shape, opts, single):
    """MoeLayer (experts checked once, buffers kept per T) gives the bits of route_permute + forward."""
    T, H, E, k, I = shape
    W = syn.make_weights(E, H, I, seed=5, device="cuda")
    layer = kt.MoeLayer(*W, k, single_launch=single, **opts)
    for t in (T, max(1, T // 3), T):   # a second T, then the first again (kept buffers)
        hidden = syn.make_hidden(t, H, seed=t, device="cuda")
        g = torch.Generator(device="cpu").manual_seed(t)
        logits = torch.randn(t, E, generator=g).cuda()
        out, ids, w = layer(hidden, logits)
        ids_r, w_r, *_ = kt.route_permute(logits, k)
        ref = kt.forward(hidden, ids_r, w_r, *W, **opts)
        torch.cuda.synchronize()
        assert torch.equal(ids, ids_r) and torch.equal(w, w_r)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), t
