"""GPU: layerwise prefill (double-buffered host -> device expert streaming).

The streamed result must be bit-identical to calling route + forward layer
by layer with device-resident weights, and to the serialized control
("upload all experts -> compute -> synchronise" per layer).  Each of those
per-layer forwards is the oracle-checked path; a one-layer streamed prefill
on generator inputs is compared with the oracle directly.  (A multi-layer
chain is not compared with an oracle chain: the two chains' inputs diverge
after layer 0 by bf16 rounding, and MXFP8 requantisation turns that into
code flips, so the gap grows with depth for reasons unrelated to either
implementation.)  A copy failure injected on the host must drain both
streams and surface as an error, leaving the context usable.
"""
import numpy as np
import pytest
import torch

import mxfp4_weight_moe_gb300 as kt
import oracle as O
from mxfp4_weight_moe_gb300 import synthetic as syn

from helpers import OUT_RTOL, bf16_bits_np, bf16_to_f64, normwise_rel

pytestmark = pytest.mark.gpu

L, T, H, I, E, K = 3, 64, 256, 256, 8, 2


def _layers():
    weights, packs, logits = [], [], []
    for l in range(L):
        W = syn.make_weights(E, H, I, seed=100 + l, device="cpu")
        weights.append(W)
        packs.append(kt.Layerwise.pack(*W))
        logits.append(syn.make_logits(T, E, "zipf", seed=l, device="cuda"))
    return weights, packs, logits


def test_layerwise_matches_sequential_and_serialized():
    weights, packs, logits = _layers()
    hidden = syn.make_hidden(T, H, 0, device="cuda")
    lw = kt.Layerwise(packs, H, I, E, K, T_max=T)
    try:
        streamed = lw.prefill(hidden, logits)
        serial = lw.prefill(hidden, logits, serialized=True)
        torch.cuda.synchronize()
    finally:
        lw.close()
    h = hidden
    for l in range(L):
        ids, w, *_ = kt.route_permute(logits[l], K)
        h = kt.forward(h, ids, w, *[t.cuda() for t in weights[l]])
    torch.cuda.synchronize()
    assert torch.equal(streamed.view(torch.int16), h.view(torch.int16))
    assert torch.equal(serial.view(torch.int16), h.view(torch.int16))


def test_layerwise_single_layer_matches_oracle():
    weights, packs, logits = _layers()
    hidden = syn.make_hidden(T, H, 0, device="cuda")
    lw = kt.Layerwise(packs[:1], H, I, E, K, T_max=T)
    try:
        out = lw.prefill(hidden, logits[:1])
        torch.cuda.synchronize()
    finally:
        lw.close()
    ids, w = O.route(logits[0].cpu().numpy(), K)
    ref = O.moe_forward(bf16_bits_np(hidden), ids, w, *[t.numpy() for t in weights[0]], want=("out_f64",))
    rel = normwise_rel(bf16_to_f64(bf16_bits_np(out)), ref["out_f64"])
    assert rel.max() <= OUT_RTOL, rel.max()


def test_layerwise_copy_failure_is_reported_and_recoverable():
    weights, packs, logits = _layers()
    hidden = syn.make_hidden(T, H, 0, device="cuda")
    lw = kt.Layerwise(packs, H, I, E, K, T_max=T)
    try:
        lw.inject_copy_failure(1)
        with pytest.raises(kt.KTError) as ei:
            lw.prefill(hidden, logits)
        assert ei.value.status == -4
        lw.inject_copy_failure(-1)
        again = lw.prefill(hidden, logits)
        ref = lw.prefill(hidden, logits, serialized=True)
        torch.cuda.synchronize()
        assert torch.equal(again.view(torch.int16), ref.view(torch.int16))
    finally:
        lw.close()


def test_layerwise_timing_hook_reports_every_layer():
    weights, packs, logits = _layers()
    hidden = syn.make_hidden(T, H, 0, device="cuda")
    lw = kt.Layerwise(packs, H, I, E, K, T_max=T)
    try:
        lw.enable_timing(True)
        lw.prefill(hidden, logits)
        t = lw.timing()
        lw.enable_timing(False)
    finally:
        lw.close()
    assert len(t["layers"]) == L
    for copy_ms, compute_ms in t["layers"]:
        assert copy_ms > 0 and compute_ms > 0
    assert t["span_ms"] >= max(c for _, c in t["layers"])


@pytest.mark.slow
def test_layerwise_dsv4_shaped_three_layers_match_per_layer_forwards():
    # the DeepSeek-V4-Flash-shaped layer (H=4096, E=256, top-6, I=2048) that the 43-layer workload streams
    Ld, Td, Hd, Id, Ed, Kd = 3, 512, 4096, 2048, 256, 6
    hidden = syn.make_hidden(Td, Hd, 0, device="cuda")
    logits = [syn.make_logits(Td, Ed, "zipf", seed=l, device="cuda") for l in range(Ld)]
    packs = []
    for l in range(Ld):
        W = syn.make_weights(Ed, Hd, Id, seed=1000 * l, device="cuda")
        packs.append(kt.Layerwise.pack(*[t.cpu() for t in W]))
        del W
    lw = kt.Layerwise(packs, Hd, Id, Ed, Kd, T_max=Td)
    try:
        streamed = lw.prefill(hidden, logits).clone()
        torch.cuda.synchronize()
    finally:
        lw.close()
    off = kt.Layerwise.pack_offsets(Hd, Id, Ed)
    shapes = ((Ed, 2 * Id, Hd // 2), (Ed, 2 * Id, Hd // 32), (Ed, Hd, Id // 2), (Ed, Hd, Id // 32))
    h = hidden
    for l in range(Ld):
        dev_pack = packs[l].cuda()
        W = [dev_pack[o:o + int(np.prod(s))].view(*s) for o, s in zip(off, shapes)]
        ids, w, *_ = kt.route_permute(logits[l], Kd)
        h = kt.forward(h, ids, w, *W)
        torch.cuda.synchronize()
        del W, dev_pack
    assert torch.equal(streamed.view(torch.int16), h.view(torch.int16))


def test_layerwise_zero_copy_matches_streamed():
    # the GEMMs read each layer's experts in place from the pinned host packs: results are those of the
    # double-buffered device-slot schedule, bit for bit
    weights, packs, logits = _layers()
    hidden = syn.make_hidden(T, H, 0, device="cuda")
    lw = kt.Layerwise(packs, H, I, E, K, T_max=T)
    zc = kt.Layerwise(packs, H, I, E, K, T_max=T, zero_copy=True)
    try:
        ref = lw.prefill(hidden, logits).clone()
        zc.enable_timing(True)
        got = zc.prefill(hidden, logits).clone()
        t = zc.timing()
        serial = zc.prefill(hidden, logits, serialized=True).clone()
        torch.cuda.synchronize()
    finally:
        lw.close()
        zc.close()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(serial.view(torch.int16), ref.view(torch.int16))
    assert all(c == 0.0 and m > 0 for c, m in t["layers"])
