"""fp64 CPU oracle of the fused MXFP4-weight MoE layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
(``--impl reference``) leg may import this package.  It wraps the plain C
implementation in ``mx_oracle.c`` (built with gcc + OpenMP into
``oracle/_build/``) and shares no code with the CUDA library.

Each function follows the step of the layer named in its docstring; the
element formats are the OCP MX v1.0 ones that "MXFP4" and "MXFP8" name on the
pages ("Kimi-K3 SM120 FlashInfer MXFP4 MoE", Goal; issue 2172, Environment).
Every function here is pinned by ``tests/test_oracle_pins.py`` against tables,
closed forms, library routines and brute force (see that file).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# MXO_ORACLE_SRC lets tests/test_oracle_mutants.py build a copy of the oracle
# with one planted mistake and check that the pins reject it.
_SRC = os.environ.get("MXO_ORACLE_SRC", os.path.join(_HERE, "mx_oracle.c"))
_OUT_DIR = os.path.join(_HERE, "_build") if "MXO_ORACLE_SRC" not in os.environ else os.path.dirname(_SRC)
_LIB_PATH = os.path.join(_OUT_DIR, "libmx_oracle.so")
_lock = threading.Lock()
_lib = None

MXO_OK = 0


def build(force: bool = False) -> str:
    """Compile mx_oracle.c into oracle/_build/libmx_oracle.so (gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(t):
    return ctypes.POINTER(t)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            c_u8p, c_u16p, c_i32p = _P(ctypes.c_uint8), _P(ctypes.c_uint16), _P(ctypes.c_int32)
            c_f32p, c_f64p = _P(ctypes.c_float), _P(ctypes.c_double)
            L.mxo_e2m1_value.argtypes = [ctypes.c_uint]
            L.mxo_e2m1_value.restype = ctypes.c_double
            L.mxo_e8m0_value.argtypes = [ctypes.c_uint]
            L.mxo_e8m0_value.restype = ctypes.c_double
            L.mxo_e4m3_value.argtypes = [ctypes.c_uint]
            L.mxo_e4m3_value.restype = ctypes.c_double
            L.mxo_e4m3_encode.argtypes = [ctypes.c_double]
            L.mxo_e4m3_encode.restype = ctypes.c_uint
            L.mxo_mx_block_exponent.argtypes = [ctypes.c_double, ctypes.c_int]
            L.mxo_mx_block_exponent.restype = ctypes.c_int
            L.mxo_quant_mxfp8.argtypes = [c_f64p, ctypes.c_int, c_u8p, c_u8p]
            L.mxo_quant_mxfp8.restype = ctypes.c_int
            L.mxo_bf16_value.argtypes = [ctypes.c_uint16]
            L.mxo_bf16_value.restype = ctypes.c_double
            L.mxo_bf16_round.argtypes = [ctypes.c_double]
            L.mxo_bf16_round.restype = ctypes.c_uint16
            L.mxo_quant_rows_bf16.argtypes = [c_u16p, ctypes.c_int, ctypes.c_int, c_u8p, c_u8p]
            L.mxo_quant_rows_bf16.restype = ctypes.c_int
            L.mxo_route.argtypes = [c_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, c_i32p, c_f32p]
            L.mxo_route.restype = ctypes.c_int
            L.mxo_permute.argtypes = [c_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, c_i32p, c_i32p, c_i32p]
            L.mxo_permute.restype = ctypes.c_int
            L.mxo_gemm_mxfp8_mxfp4.argtypes = [c_u8p, c_u8p, ctypes.c_int, ctypes.c_int, c_u8p, c_u8p,
                                              ctypes.c_int, c_f64p]
            L.mxo_gemm_mxfp8_mxfp4.restype = ctypes.c_int
            L.mxo_moe_forward_tokens.argtypes = [
                c_u16p, ctypes.c_int, ctypes.c_int, c_i32p, c_f32p, ctypes.c_int,
                c_u8p, c_u8p, c_u8p, c_u8p, ctypes.c_int, ctypes.c_int,
                c_i32p, ctypes.c_int, c_u16p, c_f64p, c_u8p, c_u8p, c_f64p, ctypes.c_int]
            L.mxo_moe_forward_tokens.restype = ctypes.c_int
            L.mxo_moe_forward_tokens_ex.argtypes = L.mxo_moe_forward_tokens.argtypes + [
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double]
            L.mxo_moe_forward_tokens_ex.restype = ctypes.c_int
            L.mxo_max_threads.argtypes = []
            L.mxo_max_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check(rc: int, what: str):
    if rc < 0:
        raise RuntimeError(f"oracle {what} failed with status {rc}")
    return rc


# ---------------------------------------------------------------- formats
def e2m1_value(nibble: int) -> float:
    """Value of one e2m1 (FP4) nibble (OCP MX v1.0 FP4 element)."""
    return lib().mxo_e2m1_value(int(nibble))


def e8m0_value(s: int) -> float:
    """Value 2^(s-127) of one e8m0 scale byte; NaN for 255."""
    return lib().mxo_e8m0_value(int(s))


def e4m3_value(code: int) -> float:
    """Value of one OCP E4M3FN code."""
    return lib().mxo_e4m3_value(int(code))


def e4m3_encode(x: float) -> int:
    """e4m3 code of x: round-to-nearest-even, saturating at +-448."""
    return int(lib().mxo_e4m3_encode(float(x)))


def block_exponent(amax: float, emax_elem: int) -> int:
    """Shared MX exponent floor(log2 amax) - emax_elem, clamped to [-127, 127]."""
    return int(lib().mxo_mx_block_exponent(float(amax), int(emax_elem)))


def quant_mxfp8(x: np.ndarray):
    """MXFP8 quantisation of a 1-D array (len % 32 == 0) -> (codes u8, scales u8)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    codes = np.empty(x.shape[0], np.uint8)
    scales = np.empty(x.shape[0] // 32, np.uint8)
    _check(lib().mxo_quant_mxfp8(_ptr(x, ctypes.c_double), x.shape[0], _ptr(codes, ctypes.c_uint8),
                                 _ptr(scales, ctypes.c_uint8)), "quant_mxfp8")
    return codes, scales


def bf16_value(bits: int) -> float:
    return lib().mxo_bf16_value(int(bits))


def bf16_round(x: float) -> int:
    """bf16 bit pattern of x (round-to-nearest-even, directly from fp64)."""
    return int(lib().mxo_bf16_round(float(x)))


def quant_rows_bf16(x_bits: np.ndarray):
    """Activation quantisation step: MXFP8 of each bf16 row -> (codes [R, C], scales [R, C/32])."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, C = x_bits.shape
    codes = np.empty((R, C), np.uint8)
    scales = np.empty((R, C // 32), np.uint8)
    _check(lib().mxo_quant_rows_bf16(_ptr(x_bits, ctypes.c_uint16), R, C, _ptr(codes, ctypes.c_uint8),
                                     _ptr(scales, ctypes.c_uint8)), "quant_rows_bf16")
    return codes, scales


# ---------------------------------------------------------------- routing
def route(logits: np.ndarray, k: int, renormalize: bool = True):
    """Route step: top-k experts per token and their softmax gating weights."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    _check(lib().mxo_route(_ptr(logits, ctypes.c_float), T, E, k, int(bool(renormalize)),
                           _ptr(ids, ctypes.c_int32), _ptr(w, ctypes.c_float)), "route")
    return ids, w


def permute(ids: np.ndarray, E: int):
    """Permute step: (expert_offsets [E+1], perm [S], inv_perm [S], n_invalid)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    bad = _check(lib().mxo_permute(_ptr(ids, ctypes.c_int32), T, k, E, _ptr(offsets, ctypes.c_int32),
                                   _ptr(perm, ctypes.c_int32), _ptr(inv, ctypes.c_int32)), "permute")
    return offsets, perm, inv, bad


# ---------------------------------------------------------------- GEMM / layer
def gemm(a: np.ndarray, a_sf: np.ndarray, w: np.ndarray, w_sf: np.ndarray) -> np.ndarray:
    """Block-scaled MXFP8 x MXFP4 GEMM in fp64: a [M, K] e4m3, w [N, K/2] fp4x2 -> [M, N]."""
    a = np.ascontiguousarray(a, np.uint8)
    a_sf = np.ascontiguousarray(a_sf, np.uint8)
    w = np.ascontiguousarray(w, np.uint8)
    w_sf = np.ascontiguousarray(w_sf, np.uint8)
    M, K = a.shape
    N = w.shape[0]
    assert w.shape[1] * 2 == K and a_sf.shape == (M, K // 32) and w_sf.shape == (N, K // 32)
    out = np.empty((M, N), np.float64)
    _check(lib().mxo_gemm_mxfp8_mxfp4(_ptr(a, ctypes.c_uint8), _ptr(a_sf, ctypes.c_uint8), M, K,
                                      _ptr(w, ctypes.c_uint8), _ptr(w_sf, ctypes.c_uint8), N,
                                      _ptr(out, ctypes.c_double)), "gemm")
    return out


def check_fc_shapes(w13: np.ndarray, w2: np.ndarray):
    """Return (E, I, H) after checking the gated FC1 / FC2 inter sizes.

    The gated FC1 packs gate and up projections, so its inter size (rows per
    expert) must be twice FC2's inter size ("Kimi-K3 SM120 FlashInfer MXFP4
    MoE", on-device evidence: 256 vs 128 for the official test shape)."""
    E, fc1_inter, h_half = w13.shape
    E2, H, i_half = w2.shape
    fc2_inter = 2 * i_half
    if E2 != E or 2 * h_half != H:
        raise ValueError(f"w13 {tuple(w13.shape)} and w2 {tuple(w2.shape)} disagree on E or H")
    if fc1_inter != 2 * fc2_inter:
        raise ValueError(f"gated FC1 inter size {fc1_inter} must be twice the FC2 inter size "
                         f"{fc2_inter} (expected {2 * fc2_inter})")
    return E, fc2_inter, H


GATE_UP_LAYOUTS = ("halves", "interleaved")
ACTIVATIONS = ("swiglu", "swiglu_clamped")


def moe_forward(hidden_bits: np.ndarray, ids: np.ndarray, topk_w: np.ndarray,
                w13, w13_sf, w2, w2_sf, tokens=None, want=("out",), nthreads: int = 0,
                gate_up: str = "halves", activation: str = "swiglu", alpha: float = 1.702, limit: float = 7.0):
    """The whole layer for the listed tokens (default: all).

    gate_up: "halves" (w13 rows [0, I) gate, [I, 2I) up) or "interleaved"
    (row 2i gate, row 2i+1 up).  activation: "swiglu" (silu(g) * u) or
    "swiglu_clamped" (min(g, limit) * sigmoid(alpha * min(g, limit)) *
    (clamp(u, -limit, limit) + 1), the gated activation of GPT-OSS-format
    checkpoints, whose SwiGLU weight layout and parameters "Kimi-K3 SM120
    FlashInfer MXFP4 MoE", Phase 0 audit conclusions, item 4, names).

    Returns a dict with any of: "out" (bf16 bits [n, H]), "out_f64" [n, H],
    "a2" (e4m3 [n, k, I]), "a2_sf" ([n, k, I/32]), "y" (fp64 [n, k, H])."""
    hidden_bits = np.ascontiguousarray(hidden_bits, np.uint16)
    ids = np.ascontiguousarray(ids, np.int32)
    topk_w = np.ascontiguousarray(topk_w, np.float32)
    w13, w13_sf, w2, w2_sf = (np.ascontiguousarray(x, np.uint8) for x in (w13, w13_sf, w2, w2_sf))
    E, I, H = check_fc_shapes(w13, w2)
    T, k = ids.shape
    assert hidden_bits.shape == (T, H) and topk_w.shape == (T, k)
    assert w13_sf.shape == (E, 2 * I, H // 32) and w2_sf.shape == (E, H, I // 32)
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, np.int32)
    n = tokens.shape[0]
    res = {}
    out = np.empty((n, H), np.uint16) if "out" in want else None
    out_f64 = np.empty((n, H), np.float64) if "out_f64" in want else None
    a2 = np.empty((n, k, I), np.uint8) if "a2" in want else None
    a2_sf = np.empty((n, k, I // 32), np.uint8) if "a2_sf" in want else None
    y = np.empty((n, k, H), np.float64) if "y" in want else None
    _check(lib().mxo_moe_forward_tokens_ex(
        _ptr(hidden_bits, ctypes.c_uint16), T, H, _ptr(ids, ctypes.c_int32), _ptr(topk_w, ctypes.c_float), k,
        _ptr(w13, ctypes.c_uint8), _ptr(w13_sf, ctypes.c_uint8), _ptr(w2, ctypes.c_uint8),
        _ptr(w2_sf, ctypes.c_uint8), E, I, _ptr(tokens, ctypes.c_int32), n,
        _ptr(out, ctypes.c_uint16), _ptr(out_f64, ctypes.c_double), _ptr(a2, ctypes.c_uint8),
        _ptr(a2_sf, ctypes.c_uint8), _ptr(y, ctypes.c_double), int(nthreads),
        GATE_UP_LAYOUTS.index(gate_up), ACTIVATIONS.index(activation), float(alpha), float(limit)), "moe_forward")
    for name, arr in (("out", out), ("out_f64", out_f64), ("a2", a2), ("a2_sf", a2_sf), ("y", y)):
        if arr is not None:
            res[name] = arr
    return res


def max_threads() -> int:
    return int(lib().mxo_max_threads())
