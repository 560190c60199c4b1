"""GPU: the tcgen05 block-scaled grouped GEMM alone (diagnostic entry).

One-hot weights make every output an exact copy of one activation element
times its two scales, which pins the fp4 nibble order, the unpacked TMA
layout, the scale-factor layout in tensor memory and the row/column
mapping; a dense random case is then compared with the fp64 oracle GEMM.
"""
import numpy as np
import pytest
import torch

import mxfp4_weight_moe_gb300 as kt
import oracle as O
from mxfp4_weight_moe_gb300 import synthetic as syn

from helpers import e4m3_to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _finite_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38     # no NaN codes
    return c


def _one_hot_weights(E, N, K, col_of):
    nib = np.zeros((E, N, K), np.uint8)
    for e in range(E):
        for n in range(N):
            nib[e, n, col_of(e, n)] = 2          # e2m1 code 2 = 1.0
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def _run(act, act_sf, counts, w, w_sf):
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    out, ws = kt.grouped_gemm_f32(t(act), t(act_sf), t(offs), t(w), t(w_sf))
    torch.cuda.synchronize()
    err = kt.read_device_error(ws)
    return out.cpu().numpy().astype(np.float64), offs, err


@pytest.mark.parametrize("counts", [[1, 0, 2], [5, 0, 300], [16, 17, 256, 257]])
def test_one_hot_unit_scales(counts):
    rng = np.random.default_rng(11)
    E, N, K = len(counts), 256, 256
    S = int(sum(counts))
    act = _finite_codes(rng, (S, K))
    act_sf = np.full((S, K // 32), 127, np.uint8)
    col = lambda e, n: (7 * n + 3 * e + 1) % K
    w = _one_hot_weights(E, N, K, col)
    w_sf = np.full((E, N, K // 32), 127, np.uint8)
    out, offs, err = _run(act, act_sf, counts, w, w_sf)
    assert err == 0
    av = e4m3_to_f64(act)
    want = np.zeros((S, N))
    swapped = np.zeros((S, N))
    for e in range(E):
        rows = slice(offs[e], offs[e + 1])
        cols = np.array([col(e, n) for n in range(N)])
        want[rows] = av[rows][:, cols]
        swapped[rows] = av[rows][:, cols ^ 1]
    if not np.array_equal(out, want):
        hint = "looks like swapped nibbles" if np.array_equal(out, swapped) else ""
        bad = np.argwhere(out != want)
        p, n = bad[0]
        raise AssertionError(f"{len(bad)} mismatches {hint}; first at row {p} col {n}: got {out[p, n]} "
                             f"want {want[p, n]}")


def test_one_hot_random_scales():
    rng = np.random.default_rng(12)
    counts = [40, 200, 1, 129]
    E, N, K = len(counts), 384, 512
    S = sum(counts)
    act = _finite_codes(rng, (S, K))
    act_sf = rng.integers(118, 137, size=(S, K // 32)).astype(np.uint8)
    col = lambda e, n: (5 * n + 11 * e + 3) % K
    w = _one_hot_weights(E, N, K, col)
    w_sf = rng.integers(116, 139, size=(E, N, K // 32)).astype(np.uint8)
    out, offs, err = _run(act, act_sf, counts, w, w_sf)
    assert err == 0
    av = e4m3_to_f64(act)
    want = np.zeros((S, N))
    for e in range(E):
        for n in range(N):
            c = col(e, n)
            r = slice(offs[e], offs[e + 1])
            want[r, n] = av[r, c] * np.exp2(act_sf[r, c // 32].astype(np.float64) - 127) * \
                np.exp2(float(w_sf[e, n, c // 32]) - 127)
    bad = np.argwhere(out != want)
    assert len(bad) == 0, f"{len(bad)} mismatches, first {bad[:3].tolist()}: got {out[tuple(bad[0])]} " \
                          f"want {want[tuple(bad[0])]}"


def test_dense_against_oracle():
    rng = np.random.default_rng(13)
    counts = [3, 250, 0, 77, 300]
    E, N, K = len(counts), 256, 1024
    S = sum(counts)
    x = rng.standard_normal((S, K))
    # activations: an independent MXFP8 quantisation of x is not needed; any
    # finite codes + scales are valid inputs, so draw them from the oracle's
    # own quantiser of x (oracle -> GPU direction only)
    act = np.empty((S, K), np.uint8)
    act_sf = np.empty((S, K // 32), np.uint8)
    for r in range(S):
        act[r], act_sf[r] = O.quant_mxfp8(x[r])
    w, w_sf = syn.pack_mxfp4(torch.from_numpy(rng.standard_normal((E, N, K)) * 0.02))
    w, w_sf = w.numpy(), w_sf.numpy()
    out, offs, err = _run(act, act_sf, counts, w, w_sf)
    assert err == 0
    worst = 0.0
    for e in range(E):
        r = slice(offs[e], offs[e + 1])
        if offs[e + 1] == offs[e]:
            continue
        ref = O.gemm(act[r], act_sf[r], w[e], w_sf[e])
        rel = np.abs(out[r] - ref).max(axis=1) / np.abs(ref).max(axis=1)
        worst = max(worst, float(rel.max()))
    assert worst < 1e-5, worst
