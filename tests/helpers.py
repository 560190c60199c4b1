"""Shared helpers of the GPU parity tests (numpy <-> torch, tolerances)."""
import numpy as np
import torch

import oracle as O

# Output tolerance: normwise relative error per token row, max over tokens.
OUT_RTOL = 2e-2


def bf16_bits_np(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def mx_deq(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    *lead, n = codes.shape
    v = e4m3_to_f64(codes).reshape(*lead, n // 32, 32)
    return (v * np.exp2(scales.astype(np.float64) - 127.0)[..., None]).reshape(*lead, n)


def normwise_rel(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per row: max |got - ref| / max |ref|; rows with ref == 0 must be exactly 0 (inf otherwise)."""
    num = np.abs(got - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    out = np.where(den > 0, num / np.where(den > 0, den, 1.0), np.where(num > 0, np.inf, 0.0))
    return out


def ws_view(ws: torch.Tensor, off: int, nbytes: int) -> np.ndarray:
    return ws[off:off + nbytes].cpu().numpy()


def sample_tokens(ids: np.ndarray, n: int, seed: int = 0) -> np.ndarray:
    """Stratified token sample: first, last, a token of the hottest and of the
    coldest non-empty expert, the rest seeded at random."""
    T = ids.shape[0]
    if n >= T:
        return np.arange(T, dtype=np.int32)
    counts = np.bincount(ids.reshape(-1)[ids.reshape(-1) >= 0], minlength=1)
    hot = int(np.argmax(counts))
    nz = np.nonzero(counts)[0]
    cold = int(nz[np.argmin(counts[nz])])
    pick = [0, T - 1, int(np.nonzero((ids == hot).any(1))[0][0]), int(np.nonzero((ids == cold).any(1))[0][0])]
    rng = np.random.default_rng(seed)
    rest = rng.choice(T, size=min(T, n * 4), replace=False)
    for t in rest:
        if len(set(pick)) >= n:
            break
        pick.append(int(t))
    return np.array(sorted(set(pick))[:n], np.int32)


def oracle_subset(hidden_bits, ids, w, w13, w13_sf, w2, w2_sf, tokens, want=("out", "a2", "a2_sf"),
                  batch_bytes=6e9, **opts):
    """Oracle on a token subset using only the experts those tokens touch.

    w13 ... may be torch CUDA tensors; only the touched experts are copied to
    the host (ids are remapped to the compact expert list).  Tokens go in
    batches whose touched experts hold at most about batch_bytes, so that a
    sample of the 36.7 GB Kimi-K3-shaped layer never copies it all.  opts
    (gate_up, activation, alpha, limit) go to the oracle's forward."""
    E = w13.shape[0]
    per_expert = sum(t[0].numel() * t.element_size() for t in (w13, w13_sf, w2, w2_sf))
    tokens = np.asarray(tokens, np.int32)
    k = ids.shape[1]
    per_batch = max(1, int(batch_bytes // max(1, per_expert * k)))
    parts = []
    for i in range(0, tokens.shape[0], per_batch):
        tk = tokens[i:i + per_batch]
        sub_ids = ids[tk]
        ok = (sub_ids >= 0) & (sub_ids < E)
        used = np.unique(sub_ids[ok])
        remap = -np.ones(E + 1, np.int64)
        remap[used] = np.arange(used.shape[0])
        idx = torch.from_numpy(used).to(w13.device)
        W = [t.index_select(0, idx).cpu().numpy() for t in (w13, w13_sf, w2, w2_sf)]
        rid = np.where(ok, remap[np.clip(sub_ids, 0, E)], -1)
        parts.append(O.moe_forward(hidden_bits[tk], rid.astype(np.int32), w[tk], *W, want=want, **opts))
        del W
    return {key: np.concatenate([p[key] for p in parts], axis=0) for key in parts[0]}


def scale_flips_valid(a2_gpu_codes, a2_gpu_sf, a2_ref_codes, a2_ref_sf):
    """Blocks whose A2 scale bytes differ, and whether each difference is the
    power-of-two straddle that fp32 vs fp64 h can cause.

    The shared exponent is floor(log2 amax) - 8, so the two sides pick
    exponents X and X + 1 only when the block amax sits at 2^(X+9): the side
    with the lower exponent then holds amax * 2^-X just below 512, which
    saturates to the largest code 448, and the side with the higher exponent
    holds amax * 2^-(X+1) just at 256, whose code is 256.  Any other scale
    difference is a real error.  Returns (n_blocks_differing, n_invalid)."""
    g = np.asarray(a2_gpu_sf, np.int64)
    r = np.asarray(a2_ref_sf, np.int64)
    diff = np.nonzero(g != r)
    if diff[0].size == 0:
        return 0, 0
    *lead, nb = g.shape
    gc = e4m3_to_f64(a2_gpu_codes).reshape(*lead, nb, 32)
    rc = e4m3_to_f64(a2_ref_codes).reshape(*lead, nb, 32)
    bad = 0
    for idx in zip(*diff):
        lo_codes, hi_codes = (gc[idx], rc[idx]) if g[idx] < r[idx] else (rc[idx], gc[idx])
        ok = abs(int(g[idx]) - int(r[idx])) == 1 and np.abs(lo_codes).max() == 448.0 and \
            np.abs(hi_codes).max() == 256.0
        bad += 0 if ok else 1
    return int(diff[0].size), bad


def check_a2(a2_gpu_codes, a2_gpu_sf, a2_ref_codes, a2_ref_sf, max_flip_frac=1e-3):
    """A2 (requantised SwiGLU output): codes may differ by one e4m3 step on a
    small fraction of elements (fp32 vs fp64 h near a rounding boundary);
    scale bytes may differ only when the block amax straddles a power of 2
    (checked separately by scale_flips_valid)."""
    dg = mx_deq(a2_gpu_codes, a2_gpu_sf)
    dr = mx_deq(a2_ref_codes, a2_ref_sf)
    mism = (dg != dr)
    frac = mism.mean() if mism.size else 0.0
    # a mismatch must be at most one code step of the larger value
    mag = np.maximum(np.abs(dg), np.abs(dr))
    X = np.maximum(a2_gpu_sf, a2_ref_sf).astype(np.float64) - 127.0
    step = np.maximum(mag * 2.0 ** -3, np.repeat(np.exp2(X - 9.0), 32, axis=-1))
    worst = (np.abs(dg - dr) / step)[mism].max() if mism.any() else 0.0
    return frac, worst
