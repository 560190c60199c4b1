"""Pins of the fp64 CPU oracle against things other than itself.

Each test ties one oracle function to a table (tests/golden, with citations),
a closed form, a library routine (torch's float8_e4m3fn / float8_e8m0fnu
dtypes, numpy's stable sort, torch.softmax / silu, numpy matmul) or brute
force on tiny inputs.  The cases are chosen so that a plausible slip -- a
swapped nibble order, a gate/up swap, a wrong exponent bias, an off-by-one in
the block exponent, a transposed operand, an unstable permutation, a dropped
routing weight -- fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from mxfp4_weight_moe_gb300 import synthetic as syn


# ------------------------------------------------------------ helpers (independent routes)
def _golden(golden_dir, name):
    rows = []
    with open(os.path.join(golden_dir, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def e2m1_table(golden_dir):
    return {int(a): float(b) for a, b in _golden(golden_dir, "e2m1_table.txt")}


def torch_e4m3_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.double().numpy()


def torch_e8m0_decode(s: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(s, np.uint8)).view(torch.float8_e8m0fnu)
    return t.double().numpy()


def torch_e4m3_encode_sat(v: np.ndarray) -> np.ndarray:
    """RNE e4m3 encode of float32-exact values via torch, with the saturation
    to +-448 applied first (torch itself does not saturate)."""
    v = np.clip(np.asarray(v, np.float64), -448.0, 448.0).astype(np.float32)
    return torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def mxfp8_ref(x: np.ndarray):
    """Independent MXFP8 quantiser for the brute-force route (numpy frexp +
    torch's e4m3 rounding).  x [..., n] fp64 -> codes, scale bytes."""
    *lead, n = x.shape
    xb = x.reshape(*lead, n // 32, 32)
    amax = np.abs(xb).max(axis=-1)
    _, e = np.frexp(amax)
    X = np.where(amax > 0, e - 1 - 8, -127).clip(-127, 127)
    v = np.ldexp(xb, -X[..., None])
    codes = torch_e4m3_encode_sat(v).reshape(*lead, n)
    return codes, (X + 127).astype(np.uint8)


def mx_dequant_e4m3(codes, scales):
    *lead, n = codes.shape
    v = torch_e4m3_decode(codes).reshape(*lead, n // 32, 32)
    return (v * torch_e8m0_decode(scales)[..., None]).reshape(*lead, n)


def mx_dequant_fp4(packed, scales, table):
    lut = np.array([table[i] for i in range(16)], np.float64)
    lo = lut[packed & 15]
    hi = lut[packed >> 4]
    *lead, kh = packed.shape
    v = np.stack([lo, hi], axis=-1).reshape(*lead, 2 * kh)      # element 2i = low nibble
    vb = v.reshape(*lead, (2 * kh) // 32, 32)
    return (vb * torch_e8m0_decode(scales)[..., None]).reshape(*lead, 2 * kh)


def bf16_bits_np(x: torch.Tensor) -> np.ndarray:
    return x.view(torch.int16).numpy().view(np.uint16)


def rand_weights(E, H, I, seed):
    w13, w13_sf, w2, w2_sf = syn.make_weights(E, H, I, seed=seed)
    return w13.numpy(), w13_sf.numpy(), w2.numpy(), w2_sf.numpy()


def dense_layer(hidden_bits, ids, w, w13, w13_sf, w2, w2_sf, table, gate_up="halves", activation="swiglu",
                alpha=1.702, limit=7.0):
    """Brute force of the whole layer on dequantised dense matrices (torch's
    silu / clamp / sigmoid for the gated activation)."""
    T, H = hidden_bits.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    x = torch.from_numpy(hidden_bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    a_codes, a_sf = mxfp8_ref(x)
    a = mx_dequant_e4m3(a_codes, a_sf)
    W13 = mx_dequant_fp4(w13, w13_sf, table)     # [E, 2I, H]
    W2 = mx_dequant_fp4(w2, w2_sf, table)        # [E, H, I]
    out = np.zeros((T, H))
    a2s = np.zeros((T, ids.shape[1], I), np.uint8)
    for t in range(T):
        for j in range(ids.shape[1]):
            e = ids[t, j]
            if e < 0 or e >= E:
                continue
            acc = W13[e] @ a[t]
            if gate_up == "halves":
                g, u = torch.from_numpy(acc[:I]), torch.from_numpy(acc[I:])
            else:
                g, u = torch.from_numpy(acc[0::2].copy()), torch.from_numpy(acc[1::2].copy())
            if activation == "swiglu":
                h = (torch.nn.functional.silu(g) * u).numpy()
            else:
                gc = torch.clamp(g, max=limit)
                uc = torch.clamp(u, min=-limit, max=limit)
                h = (gc * torch.sigmoid(alpha * gc) * (uc + 1.0)).numpy()
            c2, s2 = mxfp8_ref(h)
            a2s[t, j] = c2
            y = W2[e] @ mx_dequant_e4m3(c2, s2)
            out[t] += float(w[t, j]) * y
    return out, a2s


# ------------------------------------------------------------ formats
def test_e2m1_table(golden_dir):
    table = e2m1_table(golden_dir)
    assert len(table) == 16
    for n in range(16):
        v = O.e2m1_value(n)
        assert v == table[n] and math.copysign(1.0, v) == math.copysign(1.0, table[n]), n


def test_e8m0_all_bytes_against_torch():
    s = np.arange(256, dtype=np.uint8)
    ref = torch_e8m0_decode(s)
    for b in range(255):
        assert O.e8m0_value(b) == ref[b] == math.ldexp(1.0, b - 127), b
    assert math.isnan(O.e8m0_value(255)) and math.isnan(ref[255])


def test_e4m3_all_codes_against_torch():
    ref = torch_e4m3_decode(np.arange(256, dtype=np.uint8))
    for c in range(256):
        v = O.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), c


def test_e4m3_anchor_values(golden_dir):
    for code, val in _golden(golden_dir, "e4m3_anchors.txt"):
        c = int(code, 16)
        v = O.e4m3_value(c)
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val)), code


def test_e4m3_encode_roundtrip_all_finite_codes():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert O.e4m3_encode(O.e4m3_value(c)) == c, hex(c)


def test_e4m3_encode_ties_and_random_against_torch():
    finite = [O.e4m3_value(c) for c in range(0x7F)]          # 0 .. 448 ascending
    mids = [(finite[i] + finite[i + 1]) / 2 for i in range(len(finite) - 1)]
    rng = np.random.default_rng(0)
    rand = (rng.standard_normal(4000) * np.exp2(rng.integers(-12, 9, 4000))).astype(np.float32)
    vals = np.concatenate([np.array(mids), -np.array(mids), rand.astype(np.float64)])
    ref = torch_e4m3_encode_sat(vals)
    got = np.array([O.e4m3_encode(v) for v in vals], np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_saturates():
    for x in (448.0, 449.0, 464.0, 465.0, 480.0, 1e6, 1e300):
        assert O.e4m3_encode(x) == 0x7E
        assert O.e4m3_encode(-x) == 0xFE
    assert O.e4m3_encode(-0.0) == 0x80 and O.e4m3_encode(-1e-30) == 0x80
    assert O.e4m3_encode(float("nan")) == 0x7F


def test_block_exponent_closed_forms():
    assert O.block_exponent(1.0, 8) == -8
    assert O.block_exponent(448.0, 8) == 0
    assert O.block_exponent(511.99, 8) == 0
    assert O.block_exponent(512.0, 8) == 1
    assert O.block_exponent(0.0, 8) == -127
    assert O.block_exponent(2.0 ** -140, 8) == -127
    assert O.block_exponent(2.0 ** 200, 8) == 127
    assert O.block_exponent(6.0, 2) == 0          # e2m1: 6 = 1.5 * 2^2
    assert O.block_exponent(0.046, 2) == -7


def test_mxfp8_quantiser_invariants():
    rng = np.random.default_rng(1)
    for trial in range(200):
        x = rng.standard_normal(64) * np.exp2(rng.integers(-20, 20))
        codes, sc = O.quant_mxfp8(x)
        for b in range(2):
            X = int(sc[b]) - 127
            blk = x[32 * b:32 * b + 32]
            assert X == math.frexp(np.abs(blk).max())[1] - 1 - 8
            deq = np.array([O.e4m3_value(c) for c in codes[32 * b:32 * b + 32]]) * 2.0 ** X
            for xi, di in zip(blk, deq):
                v = abs(xi) * 2.0 ** -X
                ulp = 2.0 ** -9 if v < 2.0 ** -6 else 2.0 ** (math.frexp(v)[1] - 1 - 3)
                if v <= 448:
                    assert abs(xi - di) <= 0.5 * ulp * 2.0 ** X + 1e-300
        # scaling a block by 2^n moves the scale byte by n and keeps the codes
        n = int(rng.integers(-5, 6))
        c2, s2 = O.quant_mxfp8(x * 2.0 ** n)
        np.testing.assert_array_equal(c2, codes)
        np.testing.assert_array_equal(s2.astype(int), sc.astype(int) + n)


def test_mxfp8_quantiser_matches_independent_route():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((16, 256)) * 3).astype(np.float32).astype(np.float64)
    x[3, :32] = 0.0                    # all-zero block -> scale byte 0
    x[4, 32:64] = 1e-30                # tiny block
    want_c, want_s = mxfp8_ref(x)
    for r in range(16):
        c, s = O.quant_mxfp8(x[r])
        np.testing.assert_array_equal(c, want_c[r])
        np.testing.assert_array_equal(s, want_s[r])
    assert O.quant_mxfp8(x[3])[1][0] == 0


def test_bf16_round():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(5000) * np.exp2(rng.integers(-130, 120, 5000))).astype(np.float32)
    ref = bf16_bits_np(torch.from_numpy(v).to(torch.bfloat16))
    got = np.array([O.bf16_round(float(a)) for a in v], np.uint16)
    np.testing.assert_array_equal(got, ref)
    # directly from fp64 (no double rounding through float32):
    assert O.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert O.bf16_round(1.0 + 2.0 ** -8) == 0x3F80          # tie -> even
    assert O.bf16_round(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie -> even (up)
    for bits in (0x0000, 0x3F80, 0xBF80, 0x0001, 0x7F7F, 0xC2F6):
        assert O.bf16_round(O.bf16_value(bits)) == bits


def test_quant_rows_bf16_matches_independent_route():
    h = syn.make_hidden(8, 256, seed=4)
    bits = bf16_bits_np(h)
    c, s = O.quant_rows_bf16(bits)
    wc, ws = mxfp8_ref(h.double().numpy())
    np.testing.assert_array_equal(c, wc)
    np.testing.assert_array_equal(s, ws)


# ------------------------------------------------------------ routing / permutation
def route_ref(logits, k, renorm):
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))[:k]
        ids[t] = order
        if renorm:
            p = torch.softmax(torch.from_numpy(logits[t, order].astype(np.float64)), 0)
        else:
            p = torch.softmax(torch.from_numpy(logits[t].astype(np.float64)), 0)[order]
        w[t] = p.float().numpy()
    return ids, w


@pytest.mark.parametrize("renorm", [True, False])
def test_route_against_sort_and_softmax(renorm):
    logits = syn.make_logits(64, 37, "normal", seed=5).numpy()
    logits[0, :] = 0.5                       # all tied: lowest indices first
    logits[1, 3] = logits[1, 7] = 9.0        # a tie at the top
    ids, w = O.route(logits, 5, renorm)
    rid, rw = route_ref(logits, 5, renorm)
    np.testing.assert_array_equal(ids, rid)
    assert list(ids[0]) == [0, 1, 2, 3, 4] and list(ids[1][:2]) == [3, 7]
    ulp = np.spacing(np.abs(rw))
    assert np.all(np.abs(w.astype(np.float64) - rw.astype(np.float64)) <= ulp)
    if renorm:
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-6)


def test_route_k_equals_E_picks_all():
    logits = syn.make_logits(3, 2, "normal", seed=0).numpy()
    ids, w = O.route(logits, 2, True)
    assert sorted(ids[0]) == [0, 1]


def permute_ref(ids, E):
    flat = ids.reshape(-1)
    key = np.where((flat >= 0) & (flat < E), flat, E)
    order = np.argsort(key, kind="stable")
    counts = np.bincount(key, minlength=E + 1)[:E]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    nvalid = offsets[-1]
    perm = np.full(flat.shape[0], -1, np.int32)
    perm[:nvalid] = order[:nvalid]
    inv = np.full(flat.shape[0], -1, np.int32)
    inv[order[:nvalid]] = np.arange(nvalid)
    return offsets, perm, inv


def test_permute_against_stable_sort():
    rng = np.random.default_rng(6)
    ids = rng.integers(0, 11, size=(200, 3)).astype(np.int32)
    ids[5, 1] = 11       # out of range -> skipped
    ids[7, 0] = -1
    off, perm, inv, bad = O.permute(ids, 11)
    roff, rperm, rinv = permute_ref(ids, 11)
    np.testing.assert_array_equal(off, roff)
    np.testing.assert_array_equal(perm, rperm)
    np.testing.assert_array_equal(inv, rinv)
    assert bad == 2 and off[-1] == ids.size - 2


def test_permute_counts_and_empty_expert():
    cfg = syn.CONFIGS["small_T32"]
    lg = syn.make_logits(cfg.T, cfg.E, cfg.logits, seed=0).numpy()
    ids, _ = O.route(lg, cfg.k)
    off, perm, inv, bad = O.permute(ids, cfg.E)
    assert bad == 0 and off[-1] == cfg.T * cfg.k
    counts = np.diff(off)
    assert counts[0] == cfg.T                       # the hot expert receives every token
    assert counts[cfg.E - 1] == 0 and off[cfg.E - 1] == off[cfg.E]   # the cold one none
    assert np.all(inv[perm] == np.arange(cfg.T * cfg.k))


# ------------------------------------------------------------ GEMM and layer
def test_gemm_against_dense_numpy(golden_dir):
    table = e2m1_table(golden_dir)
    rng = np.random.default_rng(7)
    M, N, K = 7, 9, 96
    x = rng.standard_normal((M, K))
    a, a_sf = mxfp8_ref(x)
    w, w_sf = syn.pack_mxfp4(torch.from_numpy(rng.standard_normal((N, K)) * 0.02))
    w, w_sf = w.numpy(), w_sf.numpy()
    got = O.gemm(a, a_sf, w, w_sf)
    want = mx_dequant_e4m3(a, a_sf) @ mx_dequant_fp4(w, w_sf, table).T
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-300)
    # transposed-operand / nibble-order slips would not match:
    assert not np.allclose(got, mx_dequant_e4m3(a, a_sf) @ mx_dequant_fp4(w ^ 0x0F ^ 0xF0, w_sf, table).T)


@pytest.mark.parametrize("shape", [("tiny", None), ("custom", (4, 64, 3, 2, 64))])
def test_layer_brute_force(golden_dir, shape):
    table = e2m1_table(golden_dir)
    if shape[0] == "tiny":
        cfg = syn.CONFIGS["tiny"]
        T, H, E, k, I = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
        lg = syn.make_logits(T, E, cfg.logits, seed=0).numpy()
    else:
        T, H, E, k, I = shape[1]
        lg = syn.make_logits(T, E, "normal", seed=8).numpy()
    hidden = bf16_bits_np(syn.make_hidden(T, H, seed=8))
    w13, w13_sf, w2, w2_sf = rand_weights(E, H, I, seed=8)
    ids, w = O.route(lg, k)
    res = O.moe_forward(hidden, ids, w, w13, w13_sf, w2, w2_sf, want=("out", "out_f64", "a2"))
    want, want_a2 = dense_layer(hidden, ids, w, w13, w13_sf, w2, w2_sf, table)
    np.testing.assert_array_equal(res["a2"], want_a2)
    np.testing.assert_allclose(res["out_f64"], want, rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(res["out"], np.array([[O.bf16_round(v) for v in row] for row in res["out_f64"]]))


def test_layer_one_hot_closed_form():
    """E = k = T = 1, H = 64, I = 32, every weight row one-hot with scale 2^0.

    gate[n] = c_n * x[g(n)], up[n] = c'_n * x[u(n)] (gate rows first, up rows
    second), h = silu(gate) * up, y[m] = d_m * A2[r(m)]; x is chosen so that
    its MXFP8 quantisation is exact.  Only the e4m3 rounding of h goes through
    a library routine (torch)."""
    H, I = 64, 32
    vals = [(i % 7 - 3) * 0.25 for i in range(H)]
    x = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).reshape(1, H)
    fp4_code = {1.0: 2, 1.5: 3, -2.0: 12, 0.5: 1, 3.0: 5, -1.0: 10}
    cs = [1.0, 1.5, -2.0, 0.5, 3.0, -1.0]
    g_col = [(3 * n + 1) % H for n in range(I)]
    u_col = [(5 * n + 2) % H for n in range(I)]
    r_col = [(7 * m + 3) % I for m in range(H)]
    c_g = [cs[n % 6] for n in range(I)]
    c_u = [cs[(n + 2) % 6] for n in range(I)]
    d = [cs[(m + 4) % 6] for m in range(H)]

    nib13 = np.zeros((1, 2 * I, H), np.uint8)
    for n in range(I):
        nib13[0, n, g_col[n]] = fp4_code[c_g[n]]
        nib13[0, I + n, u_col[n]] = fp4_code[c_u[n]]
    nib2 = np.zeros((1, H, I), np.uint8)
    for m in range(H):
        nib2[0, m, r_col[m]] = fp4_code[d[m]]
    pack = lambda nib: (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    w13, w2 = pack(nib13), pack(nib2)
    w13_sf = np.full((1, 2 * I, H // 32), 127, np.uint8)
    w2_sf = np.full((1, H, I // 32), 127, np.uint8)
    ids = np.zeros((1, 1), np.int32)
    tw = np.ones((1, 1), np.float32)
    res = O.moe_forward(bf16_bits_np(x), ids, tw, w13, w13_sf, w2, w2_sf, want=("out", "out_f64", "a2"))

    gate = np.array([c_g[n] * vals[g_col[n]] for n in range(I)])
    up = np.array([c_u[n] * vals[u_col[n]] for n in range(I)])
    h = gate / (1.0 + np.exp(-gate)) * up
    codes, sc = mxfp8_ref(h.reshape(1, I))
    a2 = mx_dequant_e4m3(codes, sc)[0]
    y = np.array([d[m] * a2[r_col[m]] for m in range(H)])
    # +0 and -0 encode the same value (0x00 / 0x80); a block sum of exact
    # zeros is +0 while c * (+0) with c < 0 is -0, so compare modulo that sign.
    zsign = lambda c: np.where(c == 0x80, 0, c)
    np.testing.assert_array_equal(zsign(res["a2"][0, 0]), zsign(codes[0]))
    np.testing.assert_array_equal(res["out_f64"][0], y)
    zbits = lambda b: np.where(b == 0x8000, 0, b)
    np.testing.assert_array_equal(zbits(res["out"][0]),
                                  zbits(bf16_bits_np(torch.from_numpy(y).float().to(torch.bfloat16))))
    # swapping the gate and up halves changes the answer
    h_swapped = up / (1.0 + np.exp(-up)) * gate
    assert not np.allclose(h, h_swapped)


def _small_case(seed=9, T=6, H=64, E=4, k=2, I=64):
    hidden = bf16_bits_np(syn.make_hidden(T, H, seed=seed))
    w13, w13_sf, w2, w2_sf = rand_weights(E, H, I, seed=seed)
    ids, w = O.route(syn.make_logits(T, E, "normal", seed=seed).numpy(), k)
    return hidden, ids, w, w13, w13_sf, w2, w2_sf


def test_layer_token_order_invariance():
    hidden, ids, w, *W = _small_case()
    ref = O.moe_forward(hidden, ids, w, *W)["out"]
    p = np.random.default_rng(0).permutation(hidden.shape[0])
    got = O.moe_forward(hidden[p], ids[p], w[p], *W)["out"]
    np.testing.assert_array_equal(got, ref[p])


def test_layer_zero_weights_and_zero_gates():
    hidden, ids, w, w13, w13_sf, w2, w2_sf = _small_case()
    zero = O.moe_forward(hidden, ids, w, np.zeros_like(w13), w13_sf, w2, w2_sf)["out"]
    assert np.all(zero == 0)
    zero2 = O.moe_forward(hidden, ids, w, w13, w13_sf, np.zeros_like(w2), w2_sf)["out"]
    assert np.all(zero2 == 0)
    zero3 = O.moe_forward(hidden, ids, np.zeros_like(w), w13, w13_sf, w2, w2_sf)["out"]
    assert np.all((zero3 & 0x7FFF) == 0)


def test_layer_duplicate_expert_equals_single():
    hidden, ids, w, *W = _small_case(k=1)
    single = O.moe_forward(hidden, ids, np.ones_like(w), *W, want=("out_f64",))["out_f64"]
    dup = O.moe_forward(hidden, np.repeat(ids, 2, axis=1), np.full((ids.shape[0], 2), 0.5, np.float32), *W,
                        want=("out_f64",))["out_f64"]
    np.testing.assert_array_equal(dup, single)


def test_layer_invalid_ids_contribute_nothing():
    hidden, ids, w, *W = _small_case()
    bad = ids.copy()
    bad[:, 1] = 99
    got = O.moe_forward(hidden, bad, w, *W, want=("out_f64",))["out_f64"]
    only0 = O.moe_forward(hidden, ids[:, :1], w[:, :1], *W, want=("out_f64",))["out_f64"]
    np.testing.assert_array_equal(got, only0)


def test_layer_token_subset_is_exact():
    hidden, ids, w, *W = _small_case()
    full = O.moe_forward(hidden, ids, w, *W)["out"]
    sub = O.moe_forward(hidden, ids, w, *W, tokens=np.array([4, 0, 2], np.int32))["out"]
    np.testing.assert_array_equal(sub, full[[4, 0, 2]])


def test_fc1_is_twice_fc2_inter(golden_dir):
    (T, H, E, k, I, fc1, fc2, ok), = [list(map(int, r)) for r in _golden(golden_dir, "fc_inter_sizes.txt")]
    assert fc1 == 2 * fc2 == 2 * I and ok == 1
    w13 = np.zeros((E, fc1, H // 2), np.uint8)
    w2 = np.zeros((E, H, fc2 // 2), np.uint8)
    assert O.check_fc_shapes(w13, w2) == (E, I, H)
    with pytest.raises(ValueError, match=r"256"):
        O.check_fc_shapes(np.zeros((E, fc2, H // 2), np.uint8), w2)      # non-gated 128 rows
    cfg = syn.CONFIGS["tiny"]
    assert (cfg.T, cfg.H, cfg.E, cfg.k, cfg.I) == (T, H, E, k, I)


# ------------------------------------------------------------ gate/up layout and activation variants
# The interleaved gate/up rows and the clamped SwiGLU of GPT-OSS-format checkpoints ("Kimi-K3 SM120
# FlashInfer MXFP4 MoE", Phase 0 audit conclusions, item 4): w13 row 2i is gate i and row 2i+1 up i;
# h = min(g, L) * sigmoid(alpha * min(g, L)) * (clamp(u, -L, L) + 1).
@pytest.mark.parametrize("gate_up,activation,limit", [
    ("interleaved", "swiglu", 7.0),
    ("halves", "swiglu_clamped", 0.1),        # a small limit clamps most gate and up values
    ("interleaved", "swiglu_clamped", 0.1),
    ("interleaved", "swiglu_clamped", 7.0),
])
def test_layer_variants_brute_force(golden_dir, gate_up, activation, limit):
    table = e2m1_table(golden_dir)
    T, H, E, k, I = 4, 64, 3, 2, 64
    lg = syn.make_logits(T, E, "normal", seed=8).numpy()
    hidden = bf16_bits_np(syn.make_hidden(T, H, seed=8))
    w13, w13_sf, w2, w2_sf = rand_weights(E, H, I, seed=8)
    w13_sf = (w13_sf.astype(np.int32) + 4).astype(np.uint8)    # x16: gate / up values of order 1, so L = 0.1 bites
    ids, w = O.route(lg, k)
    kw = dict(gate_up=gate_up, activation=activation, alpha=1.702, limit=limit)
    res = O.moe_forward(hidden, ids, w, w13, w13_sf, w2, w2_sf, want=("out_f64", "a2"), **kw)
    want, want_a2 = dense_layer(hidden, ids, w, w13, w13_sf, w2, w2_sf, table, **kw)
    np.testing.assert_array_equal(res["a2"], want_a2)
    np.testing.assert_allclose(res["out_f64"], want, rtol=1e-10, atol=1e-12)
    # the variant is a different layer from the default one
    base = O.moe_forward(hidden, ids, w, w13, w13_sf, w2, w2_sf, want=("out_f64",))["out_f64"]
    assert not np.allclose(base, res["out_f64"])


@pytest.mark.parametrize("activation", ["swiglu", "swiglu_clamped"])
def test_interleaved_rows_equal_halves_layout(activation):
    """Interleaving the rows of a gate | up w13 (row 2i <- gate i, row 2i+1 <- up i) and reading it
    as interleaved gives exactly the halves-layout result."""
    hidden, ids, w, w13, w13_sf, w2, w2_sf = _small_case(I=64)
    I = w13.shape[1] // 2
    order = np.empty(2 * I, np.int64)
    order[0::2] = np.arange(I)
    order[1::2] = I + np.arange(I)
    kw = dict(activation=activation, alpha=1.702, limit=0.5)
    a = O.moe_forward(hidden, ids, w, w13, w13_sf, w2, w2_sf, want=("out", "a2"), gate_up="halves", **kw)
    b = O.moe_forward(hidden, ids, w, np.ascontiguousarray(w13[:, order]), np.ascontiguousarray(w13_sf[:, order]),
                      w2, w2_sf, want=("out", "a2"), gate_up="interleaved", **kw)
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["a2"], b["a2"])
    # reading the halves layout as interleaved is a different (wrong) layer
    c = O.moe_forward(hidden, ids, w, w13, w13_sf, w2, w2_sf, want=("out",), gate_up="interleaved", **kw)
    assert not np.array_equal(a["out"], c["out"])


def test_clamped_swiglu_one_hot_closed_form():
    """E = k = T = 1, H = 64, I = 32, interleaved one-hot w13 rows (row 2n gate, 2n+1 up), limit 1 so that
    gate values above 1 and up values beyond +-1 are clamped; h from the closed form in numpy."""
    H, I, L, alpha = 64, 32, 1.0, 1.702
    vals = [(i % 7 - 3) * 0.25 for i in range(H)]
    x = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).reshape(1, H)
    fp4_code = {1.0: 2, 1.5: 3, -2.0: 12, 0.5: 1, 3.0: 5, -1.0: 10, 4.0: 6, -3.0: 13}
    cs = [1.0, 1.5, -2.0, 0.5, 3.0, -1.0, 4.0, -3.0]
    g_col = [(3 * n + 1) % H for n in range(I)]
    u_col = [(5 * n + 2) % H for n in range(I)]
    r_col = [(7 * m + 3) % I for m in range(H)]
    c_g = [cs[n % 8] for n in range(I)]
    c_u = [cs[(n + 3) % 8] for n in range(I)]
    d = [cs[(m + 4) % 6] for m in range(H)]
    nib13 = np.zeros((1, 2 * I, H), np.uint8)
    for n in range(I):
        nib13[0, 2 * n, g_col[n]] = fp4_code[c_g[n]]
        nib13[0, 2 * n + 1, u_col[n]] = fp4_code[c_u[n]]
    nib2 = np.zeros((1, H, I), np.uint8)
    for m in range(H):
        nib2[0, m, r_col[m]] = fp4_code[d[m]]
    pack = lambda nib: (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    w13, w2 = pack(nib13), pack(nib2)
    w13_sf = np.full((1, 2 * I, H // 32), 127, np.uint8)
    w2_sf = np.full((1, H, I // 32), 127, np.uint8)
    res = O.moe_forward(bf16_bits_np(x), np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), w13, w13_sf, w2,
                        w2_sf, want=("out_f64", "a2"), gate_up="interleaved", activation="swiglu_clamped",
                        alpha=alpha, limit=L)
    gate = np.array([c_g[n] * vals[g_col[n]] for n in range(I)])
    up = np.array([c_u[n] * vals[u_col[n]] for n in range(I)])
    assert (gate > L).any() and (up > L).any() and (up < -L).any() and (gate < -L).any()
    gc = np.minimum(gate, L)
    uc = np.clip(up, -L, L)
    h = gc / (1.0 + np.exp(-alpha * gc)) * (uc + 1.0)
    codes, sc = mxfp8_ref(h.reshape(1, I))
    a2 = mx_dequant_e4m3(codes, sc)[0]
    y = np.array([d[m] * a2[r_col[m]] for m in range(H)])
    zsign = lambda c: np.where(c == 0x80, 0, c)
    np.testing.assert_array_equal(zsign(res["a2"][0, 0]), zsign(codes[0]))
    np.testing.assert_array_equal(res["out_f64"][0], y)
