"""GB300 (sm_103a) fused MXFP4-weight mixture-of-experts layer.

Thin Python binding over the C ABI in ``include/kt_moe.h`` (library
``_build/libkt_moe.so``, built by ``build_ext.build``).  Every step of the
layer runs in the library's CUDA kernels; this module only checks shapes,
allocates outputs/workspaces with torch and passes raw device pointers and
the current CUDA stream.  There is no CPU or torch fallback: if the library
cannot be built or loaded, every op raises.

Formats: hidden/out bf16 [T, H]; topk_ids int32 [T, k]; topk_w float32 [T, k];
w13 uint8 fp4x2 [E, 2I, H/2] (rows [0, I) gate, [I, 2I) up; element 2i in the
low nibble) + w13_sf uint8 e8m0 [E, 2I, H/32]; w2 uint8 fp4x2 [E, H, I/2] +
w2_sf uint8 e8m0 [E, H, I/32].
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import build_ext

__all__ = [
    "KTError", "lib", "route_permute", "forward", "workspace_bytes", "workspace_layout", "read_device_error",
    "grouped_gemm_f32", "Layerwise", "status_string", "check_fc_shapes", "kernel_launches", "profile_enable",
    "profile_read", "STAGES", "route_permute_noalloc", "decode", "DECODE_MAX_SLOTS", "MoeLayer",
]

KT_OK = 0
KT_DEVERR_BAD_EXPERT_ID = 0x1
KT_DEVERR_TIMEOUT_LOAD = 0x2
KT_DEVERR_TIMEOUT_MMA = 0x4
KT_DEVERR_TIMEOUT_EPI = 0x8

_lock = threading.Lock()
_lib = None


class KTError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status}) {detail}".strip())


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("err", "expert_offsets", "chunk_prefix", "perm", "inv_perm", "hist", "a1", "a1_sf", "a2", "a2_sf",
                 "y", "total")]


class MoeOptions(ctypes.Structure):
    _fields_ = [("gate_up_layout", ctypes.c_int), ("activation", ctypes.c_int), ("alpha", ctypes.c_float),
                ("limit", ctypes.c_float)]


GATE_UP_LAYOUTS = ("halves", "interleaved")
ACTIVATIONS = ("swiglu", "swiglu_clamped")

_VP, _SZ, _I = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int

_SIGNATURES = {
    "kt_status_string": ([_I], ctypes.c_char_p),
    "kt_last_error": ([], ctypes.c_char_p),
    "kt_moe_route_workspace_bytes": ([_I, _I, _I], _SZ),
    "kt_moe_route_permute": ([_VP, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP], _I),
    "kt_moe_workspace_bytes": ([_I, _I, _I, _I, _I], _SZ),
    "kt_mxfp4_moe_forward": ([_VP, _I, _I, _VP, _VP, _I, _VP, _VP, _VP, _VP, _I, _I, _VP, _VP, _SZ, _VP], _I),
    "kt_mxfp4_moe_forward_ex": ([_VP, _I, _I, _VP, _VP, _I, _VP, _VP, _VP, _VP, _I, _I, _VP, _VP, _SZ,
                                 ctypes.POINTER(MoeOptions), _VP], _I),
    "kt_mxfp4_moe_forward_routed": ([_VP, _I, _I, _VP, _VP, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _VP,
                                     _VP, _SZ, ctypes.POINTER(MoeOptions), _VP], _I),
    "kt_mxfp4_moe_decode": ([_VP, _VP, _I, _I, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ,
                             ctypes.POINTER(MoeOptions), _VP], _I),
    "kt_moe_workspace_layout": ([_I, _I, _I, _I, _I, ctypes.POINTER(WsLayout)], _I),
    "kt_moe_read_device_error": ([_VP, ctypes.POINTER(_I), _VP], _I),
    "kt_mx_gemm_workspace_bytes": ([_I, _I, _I], _SZ),
    "kt_mx_grouped_gemm_f32": ([_VP, _VP, _I, _I, _VP, _VP, _VP, _I, _I, _VP, _VP, _SZ, _VP], _I),
    "kt_layerwise_pack_bytes": ([_I, _I, _I], _SZ),
    "kt_layerwise_pack_offsets": ([_I, _I, _I, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ), ctypes.POINTER(_SZ),
                                   ctypes.POINTER(_SZ)], _I),
    "kt_layerwise_create": ([ctypes.POINTER(_VP), _I, _I, _I, _I, _I, _I, ctypes.POINTER(_VP)], _I),
    "kt_layerwise_prefill": ([_VP, _VP, ctypes.POINTER(_VP), _VP, _I, _I, _VP], _I),
    "kt_layerwise_inject_copy_failure": ([_VP, _I], _I),
    "kt_layerwise_create_zero_copy": ([ctypes.POINTER(_VP), _I, _I, _I, _I, _I, _I, ctypes.POINTER(_VP)], _I),
    "kt_layerwise_enable_timing": ([_VP, _I], _I),
    "kt_layerwise_read_timing": ([_VP, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_double)], _I),
    "kt_layerwise_destroy": ([_VP], _I),
    "kt_moe_kernel_launches": ([], ctypes.c_uint64),
    "kt_moe_profile_enable": ([_I], _I),
    "kt_moe_profile_read": ([ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I)], _I),
    "kt_moe_debug_configure": ([ctypes.c_uint64, _I], _I),
    "kt_moe_profile_enable_stages": ([ctypes.c_uint32], _I),
    "kt_moe_route_permute_noalloc": ([_VP, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP], _I),
}

KT_NOALLOC_SCRATCH_BYTES = 1 << 20
DECODE_MAX_SLOTS = 2048   # KT_DECODE_MAX_SLOTS

KT_DEBUG_WITHHOLD_STAGE = 0x1

STAGES = ("route", "permute", "quant", "fc1", "fc2", "combine")


def lib(build_if_missing: bool = True):
    """The loaded C library (built in-tree on first use if absent)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = build_ext.build() if build_if_missing else build_ext.LIB_PATH
            L = ctypes.CDLL(path)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().kt_status_string(int(status)).decode()
    except Exception:  # noqa: BLE001 - used while formatting an error
        return "KT_STATUS"


def _check(status: int, what: str):
    if status != KT_OK:
        detail = lib().kt_last_error().decode()
        raise KTError(status, what, detail)


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()   # the signatures declare c_void_p


def _stream_ptr(stream, device):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return s.cuda_stream


class _on_device:
    """Make `dev` the current CUDA device for a call (a no-op when it already is)."""
    __slots__ = ("idx", "prev")

    def __init__(self, dev: torch.device):
        self.idx = dev.index

    def __enter__(self):
        self.prev = torch.cuda.current_device()
        if self.idx is not None and self.idx != self.prev:
            torch.cuda.set_device(self.idx)

    def __exit__(self, *exc):
        if self.idx is not None and self.idx != self.prev:
            torch.cuda.set_device(self.prev)


def _need(t: torch.Tensor, name: str, dtype, ndim: int, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def check_fc_shapes(w13: torch.Tensor, w2: torch.Tensor):
    """(E, I, H) after checking that the gated FC1 inter size (rows per expert
    of w13) is twice the FC2 inter size (2 * w2.shape[2])."""
    E, fc1_inter, h_half = w13.shape
    E2, H, i_half = w2.shape
    fc2_inter = 2 * i_half
    if E2 != E or 2 * h_half != H:
        raise ValueError(f"w13 {tuple(w13.shape)} and w2 {tuple(w2.shape)} disagree on E or H")
    if fc1_inter != 2 * fc2_inter:
        raise ValueError(f"gated FC1 inter size {fc1_inter} must be twice the FC2 inter size {fc2_inter} "
                         f"(expected {2 * fc2_inter})")
    return E, fc2_inter, H


def route_permute_noalloc(logits: torch.Tensor, k: int, renormalize: bool = True, stream=None, out=None):
    """route_permute without a caller workspace: the scratch is a fixed device
    array inside the library (for callers that cannot allocate device memory;
    concurrent calls on different streams race on it).  Outputs as route_permute."""
    _need(logits, "logits", torch.float32, 2)
    T, E = logits.shape
    dev = logits.device
    if out is None:
        out = (torch.empty(T, k, dtype=torch.int32, device=dev), torch.empty(T, k, dtype=torch.float32, device=dev),
               torch.empty(E + 1, dtype=torch.int32, device=dev), torch.empty(T * k, dtype=torch.int32, device=dev),
               torch.empty(T * k, dtype=torch.int32, device=dev))
    ids, w, offsets, perm, inv = out
    with torch.cuda.device(dev):
        _check(lib().kt_moe_route_permute_noalloc(_ptr(logits), T, E, k, int(bool(renormalize)), _ptr(ids), _ptr(w),
                                                  _ptr(offsets), _ptr(perm), _ptr(inv), _stream_ptr(stream, dev)),
               "kt_moe_route_permute_noalloc")
    return ids, w, offsets, perm, inv


def workspace_bytes(T: int, H: int, I: int, E: int, k: int) -> int:
    return int(lib().kt_moe_workspace_bytes(T, H, I, E, k))


def scales_from_kstep_major(words: torch.Tensor, S: int, K: int) -> torch.Tensor:
    """Plain [S, K/32] e8m0 bytes from a workspace's K-step-major scale region
    (u32 [K/128][S4], byte b % 4 of word (b // 4, row) is block b)."""
    S4 = (S + 3) // 4 * 4
    w = words[: (K // 128) * S4 * 4].view(K // 128, S4, 4)
    return w[:, :S, :].permute(1, 0, 2).reshape(S, K // 32)


def workspace_layout(T: int, H: int, I: int, E: int, k: int) -> dict:
    L = WsLayout()
    _check(lib().kt_moe_workspace_layout(T, H, I, E, k, ctypes.byref(L)), "kt_moe_workspace_layout")
    return {n: int(getattr(L, n)) for n, _ in WsLayout._fields_}


def route_permute(logits: torch.Tensor, k: int, renormalize: bool = True, stream=None, out=None, workspace=None):
    """Top-k routing + permutation.  Returns (topk_ids, topk_w, expert_offsets, perm, inv_perm)."""
    _need(logits, "logits", torch.float32, 2)
    T, E = logits.shape
    dev = logits.device
    if out is None:
        out = (torch.empty(T, k, dtype=torch.int32, device=dev), torch.empty(T, k, dtype=torch.float32, device=dev),
               torch.empty(E + 1, dtype=torch.int32, device=dev), torch.empty(T * k, dtype=torch.int32, device=dev),
               torch.empty(T * k, dtype=torch.int32, device=dev))
    ids, w, offsets, perm, inv = out
    if workspace is None:
        nbytes = int(lib().kt_moe_route_workspace_bytes(T, E, k))
        if nbytes == 0 and T > 0:   # invalid shape: let the library report it
            _check(lib().kt_moe_route_permute(None, T, E, k, 1, None, None, None, None, None, None, 0, None),
                   "kt_moe_route_permute")
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    with _on_device(dev):
        _check(lib().kt_moe_route_permute(_ptr(logits), T, E, k, int(bool(renormalize)), _ptr(ids), _ptr(w),
                                          _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(workspace), workspace.numel(),
                                          _stream_ptr(stream, dev)), "kt_moe_route_permute")
    return ids, w, offsets, perm, inv


def forward(hidden: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor, w13: torch.Tensor,
            w13_sf: torch.Tensor, w2: torch.Tensor, w2_sf: torch.Tensor, out: torch.Tensor | None = None,
            workspace: torch.Tensor | None = None, stream=None, gate_up: str = "halves",
            activation: str = "swiglu", alpha: float = 1.702, limit: float = 7.0,
            routing: tuple | None = None) -> torch.Tensor:
    """One fused MoE layer forward; returns out (bf16 [T, H]).

    gate_up "halves" (w13 rows [0, I) gate, [I, 2I) up) or "interleaved"
    (row 2i gate i, row 2i+1 up i); activation "swiglu" (silu(g) * u) or
    "swiglu_clamped" (the clamped SwiGLU of GPT-OSS-format checkpoints, with
    alpha and limit; see kt_moe_options in kt_moe.h).  routing: the
    (expert_offsets, perm, inv_perm) that route_permute returned for these
    topk_ids, reused instead of re-derived (kt_mxfp4_moe_forward_routed)."""
    _need(hidden, "hidden", torch.bfloat16, 2)
    dev = hidden.device
    _need(topk_ids, "topk_ids", torch.int32, 2, dev)
    _need(topk_w, "topk_w", torch.float32, 2, dev)
    for name, t in (("w13", w13), ("w13_sf", w13_sf), ("w2", w2), ("w2_sf", w2_sf)):
        _need(t, name, torch.uint8, 3, dev)
    E, I, H = check_fc_shapes(w13, w2)
    T, k = topk_ids.shape
    if hidden.shape != (T, H) or topk_w.shape != (T, k):
        raise ValueError(f"hidden {tuple(hidden.shape)} / topk_w {tuple(topk_w.shape)} do not match "
                         f"T={T}, H={H}, k={k}")
    if w13_sf.shape != (E, 2 * I, H // 32) or w2_sf.shape != (E, H, I // 32):
        raise ValueError("scale tensors must be [E, 2I, H/32] and [E, H, I/32]")
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, 2, dev)
    if workspace is None:   # a caller's workspace is size-checked by the library
        workspace = torch.empty(max(workspace_bytes(T, H, I, E, k), 1), dtype=torch.uint8, device=dev)
    if routing is not None:
        offsets, perm, inv_perm = routing
        _need(offsets, "expert_offsets", torch.int32, 1, dev)
        _need(perm, "perm", torch.int32, 1, dev)
        _need(inv_perm, "inv_perm", torch.int32, 1, dev)
        if offsets.numel() != E + 1 or perm.numel() != T * k or inv_perm.numel() != T * k:
            raise ValueError("routing must be (expert_offsets [E+1], perm [T*k], inv_perm [T*k])")
        if gate_up not in GATE_UP_LAYOUTS or activation not in ACTIVATIONS:
            raise ValueError(f"gate_up must be one of {GATE_UP_LAYOUTS} and activation one of {ACTIVATIONS}")
        opts = MoeOptions(GATE_UP_LAYOUTS.index(gate_up), ACTIVATIONS.index(activation), float(alpha), float(limit))
        with _on_device(dev):
            _check(lib().kt_mxfp4_moe_forward_routed(_ptr(hidden), T, H, _ptr(topk_ids), _ptr(topk_w), k,
                                                     _ptr(offsets), _ptr(perm), _ptr(inv_perm), _ptr(w13),
                                                     _ptr(w13_sf), _ptr(w2), _ptr(w2_sf), E, I, _ptr(out),
                                                     _ptr(workspace), workspace.numel(), ctypes.byref(opts),
                                                     _stream_ptr(stream, dev)),
                   "kt_mxfp4_moe_forward_routed")
        return out
    if gate_up == "halves" and activation == "swiglu":
        with _on_device(dev):
            _check(lib().kt_mxfp4_moe_forward(_ptr(hidden), T, H, _ptr(topk_ids), _ptr(topk_w), k, _ptr(w13),
                                              _ptr(w13_sf), _ptr(w2), _ptr(w2_sf), E, I, _ptr(out),
                                              _ptr(workspace), workspace.numel(), _stream_ptr(stream, dev)),
                   "kt_mxfp4_moe_forward")
        return out
    if gate_up not in GATE_UP_LAYOUTS or activation not in ACTIVATIONS:
        raise ValueError(f"gate_up must be one of {GATE_UP_LAYOUTS} and activation one of {ACTIVATIONS}")
    opts = MoeOptions(GATE_UP_LAYOUTS.index(gate_up), ACTIVATIONS.index(activation), float(alpha), float(limit))
    with _on_device(dev):
        _check(lib().kt_mxfp4_moe_forward_ex(_ptr(hidden), T, H, _ptr(topk_ids), _ptr(topk_w), k, _ptr(w13),
                                             _ptr(w13_sf), _ptr(w2), _ptr(w2_sf), E, I, _ptr(out), _ptr(workspace),
                                             workspace.numel(), ctypes.byref(opts), _stream_ptr(stream, dev)),
               "kt_mxfp4_moe_forward_ex")
    return out


def decode(logits: torch.Tensor, hidden: torch.Tensor, k: int, w13: torch.Tensor, w13_sf: torch.Tensor,
           w2: torch.Tensor, w2_sf: torch.Tensor, renormalize: bool = True, out: torch.Tensor | None = None,
           topk: tuple | None = None, workspace: torch.Tensor | None = None, stream=None,
           gate_up: str = "halves", activation: str = "swiglu", alpha: float = 1.702, limit: float = 7.0):
    """Routing + the layer forward in ONE kernel launch (T * k <= DECODE_MAX_SLOTS).

    Same results as route_permute followed by forward.  Returns
    (out bf16 [T, H], topk_ids int32 [T, k], topk_w float32 [T, k])."""
    _need(logits, "logits", torch.float32, 2)
    dev = logits.device
    _need(hidden, "hidden", torch.bfloat16, 2, dev)
    for name, t in (("w13", w13), ("w13_sf", w13_sf), ("w2", w2), ("w2_sf", w2_sf)):
        _need(t, name, torch.uint8, 3, dev)
    E, I, H = check_fc_shapes(w13, w2)
    T = hidden.shape[0]
    if hidden.shape != (T, H) or logits.shape != (T, E):
        raise ValueError(f"hidden {tuple(hidden.shape)} / logits {tuple(logits.shape)} do not match T={T}, H={H}, "
                         f"E={E}")
    if w13_sf.shape != (E, 2 * I, H // 32) or w2_sf.shape != (E, H, I // 32):
        raise ValueError("scale tensors must be [E, 2I, H/32] and [E, H, I/32]")
    if gate_up not in GATE_UP_LAYOUTS or activation not in ACTIVATIONS:
        raise ValueError(f"gate_up must be one of {GATE_UP_LAYOUTS} and activation one of {ACTIVATIONS}")
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, 2, dev)
    if topk is None:
        topk = (torch.empty(T, k, dtype=torch.int32, device=dev), torch.empty(T, k, dtype=torch.float32, device=dev))
    ids, w = topk
    if workspace is None:
        workspace = torch.empty(max(workspace_bytes(T, H, I, E, k), 1), dtype=torch.uint8, device=dev)
    opts = MoeOptions(GATE_UP_LAYOUTS.index(gate_up), ACTIVATIONS.index(activation), float(alpha), float(limit))
    with _on_device(dev):
        _check(lib().kt_mxfp4_moe_decode(_ptr(logits), _ptr(hidden), T, H, E, k, I, int(bool(renormalize)),
                                         _ptr(w13), _ptr(w13_sf), _ptr(w2), _ptr(w2_sf), _ptr(ids), _ptr(w), _ptr(out),
                                         _ptr(workspace), workspace.numel(), ctypes.byref(opts),
                                         _stream_ptr(stream, dev)), "kt_mxfp4_moe_decode")
    return out, ids, w


def read_device_error(workspace: torch.Tensor, stream=None) -> int:
    """Device error word of the last forward/route call that used `workspace`."""
    code = ctypes.c_int(0)
    st = lib().kt_moe_read_device_error(_ptr(workspace), ctypes.byref(code), _stream_ptr(stream, workspace.device))
    if st not in (KT_OK, -6, -8):
        _check(st, "kt_moe_read_device_error")
    return code.value


def grouped_gemm_f32(act, act_sf, expert_offsets, w, w_sf, out=None, stream=None):
    """Diagnostic: the block-scaled grouped GEMM alone, fp32 out [S, N]."""
    _need(act, "act", torch.uint8, 2)
    dev = act.device
    S, K = act.shape
    E, N, _ = w.shape
    if out is None:
        out = torch.zeros(S, N, dtype=torch.float32, device=dev)
    ws = torch.empty(max(int(lib().kt_mx_gemm_workspace_bytes(S, K, E)), 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check(lib().kt_mx_grouped_gemm_f32(_ptr(act), _ptr(act_sf), S, K, _ptr(expert_offsets), _ptr(w), _ptr(w_sf),
                                            E, N, _ptr(out), _ptr(ws), ws.numel(), _stream_ptr(stream, dev)),
               "kt_mx_grouped_gemm_f32")
    return out, ws


def kernel_launches() -> int:
    """Kernels this library has launched in this process."""
    return int(lib().kt_moe_kernel_launches())


def profile_enable(enable: bool = True, stages=None):
    """Start (or stop) recording per-stage CUDA events; discards old records.
    `stages` (names from STAGES) limits the recording to those stages."""
    if stages is None:
        _check(lib().kt_moe_profile_enable(int(bool(enable))), "kt_moe_profile_enable")
        return
    mask = 0
    if enable:
        for name in stages:
            mask |= 1 << STAGES.index(name)
    _check(lib().kt_moe_profile_enable_stages(mask), "kt_moe_profile_enable_stages")


def debug_configure(wait_limit_us: int = 0, flags: int = 0):
    """Test hook: bound the GEMM barrier waits and optionally withhold a stage
    (see kt_moe_debug_configure); debug_configure() restores the defaults."""
    _check(lib().kt_moe_debug_configure(int(wait_limit_us), int(flags)), "kt_moe_debug_configure")


def profile_read() -> dict:
    """{stage: (total_ms, calls)} over the calls recorded since profile_enable()."""
    ms = (ctypes.c_double * len(STAGES))()
    calls = (ctypes.c_int * len(STAGES))()
    _check(lib().kt_moe_profile_read(ms, calls), "kt_moe_profile_read")
    return {name: (float(ms[i]), int(calls[i])) for i, name in enumerate(STAGES)}


class MoeLayer:
    """One MoE layer whose packed experts are checked once, for repeated steps.

    A call routes the step's logits and runs the layer as kt_moe_route_permute
    + kt_mxfp4_moe_forward_routed, or (single_launch=True, for batches of at
    most DECODE_MAX_SLOTS slots) as one kt_mxfp4_moe_decode launch.  Per step
    only the step's own tensors are
    checked and marshalled; workspaces and routing buffers are kept per T.
    Results are those of route_permute + forward (or decode) with the same
    options.  Returns (out, topk_ids, topk_w); the three are reused by the
    next call with the same T unless `out` is given."""

    def __init__(self, w13: torch.Tensor, w13_sf: torch.Tensor, w2: torch.Tensor, w2_sf: torch.Tensor, k: int,
                 renormalize: bool = True, gate_up: str = "halves", activation: str = "swiglu", alpha: float = 1.702,
                 limit: float = 7.0, single_launch: bool = False):
        dev = w13.device
        for name, t in (("w13", w13), ("w13_sf", w13_sf), ("w2", w2), ("w2_sf", w2_sf)):
            _need(t, name, torch.uint8, 3, dev)
        E, I, H = check_fc_shapes(w13, w2)
        if w13_sf.shape != (E, 2 * I, H // 32) or w2_sf.shape != (E, H, I // 32):
            raise ValueError("scale tensors must be [E, 2I, H/32] and [E, H, I/32]")
        if gate_up not in GATE_UP_LAYOUTS or activation not in ACTIVATIONS:
            raise ValueError(f"gate_up must be one of {GATE_UP_LAYOUTS} and activation one of {ACTIVATIONS}")
        self.E, self.I, self.H, self.k = E, I, H, int(k)
        self.renormalize = int(bool(renormalize))
        self.device = dev
        self._dev_idx = w13.get_device()
        self._weights = (w13, w13_sf, w2, w2_sf)   # keep them alive
        self._wp = tuple(t.data_ptr() for t in self._weights)
        self._opts = MoeOptions(GATE_UP_LAYOUTS.index(gate_up), ACTIVATIONS.index(activation), float(alpha),
                                float(limit))
        self._optsref = ctypes.byref(self._opts)
        self._single_launch = bool(single_launch)
        self._per_T = {}

    def _buffers(self, T: int):
        b = self._per_T.get(T)
        if b is None:
            dev, E, k, H, I = self.device, self.E, self.k, self.H, self.I
            decode = self._single_launch and T * k <= DECODE_MAX_SLOTS
            ws = torch.empty(max(workspace_bytes(T, H, I, E, k), 1), dtype=torch.uint8, device=dev)
            route = (torch.empty(T, k, dtype=torch.int32, device=dev), torch.empty(T, k, dtype=torch.float32, device=dev),
                     torch.empty(E + 1, dtype=torch.int32, device=dev), torch.empty(T * k, dtype=torch.int32, device=dev),
                     torch.empty(T * k, dtype=torch.int32, device=dev))
            rws = None if decode else torch.empty(max(int(lib().kt_moe_route_workspace_bytes(T, E, k)), 1),
                                                  dtype=torch.uint8, device=dev)
            out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
            b = (decode, ws, route, rws, out)
            self._per_T[T] = b
        return b

    def __call__(self, hidden: torch.Tensor, logits: torch.Tensor, out: torch.Tensor | None = None, stream=None):
        T = hidden.shape[0]
        if (hidden.dtype != torch.bfloat16 or logits.dtype != torch.float32 or hidden.shape != (T, self.H)
                or logits.shape != (T, self.E) or hidden.get_device() != self._dev_idx
                or logits.get_device() != self._dev_idx or not hidden.is_contiguous() or not logits.is_contiguous()):
            raise ValueError(f"hidden must be contiguous bf16 [T, {self.H}] and logits contiguous f32 [T, {self.E}] "
                             f"on {self.device}")
        decode, ws, route, rws, own_out = self._buffers(T)
        if out is None:
            out = own_out
        elif (out.dtype != torch.bfloat16 or out.shape != (T, self.H) or out.get_device() != self._dev_idx
              or not out.is_contiguous()):
            raise ValueError(f"out must be contiguous bf16 [T, {self.H}] on {self.device}")
        ids, w, offs, perm, inv = route
        with _on_device(self.device):
            self._launch(T, hidden, logits, out, decode, ws, ids, w, offs, perm, inv, rws,
                         _stream_ptr(stream, self.device))
        return out, ids, w

    def _launch(self, T, hidden, logits, out, decode, ws, ids, w, offs, perm, inv, rws, sp):
        w13, w13_sf, w2, w2_sf = self._wp
        L = lib()
        if decode:
            _check(L.kt_mxfp4_moe_decode(logits.data_ptr(), hidden.data_ptr(), T, self.H, self.E, self.k, self.I,
                                         self.renormalize, w13, w13_sf, w2, w2_sf, ids.data_ptr(), w.data_ptr(),
                                         out.data_ptr(), ws.data_ptr(), ws.numel(), self._optsref, sp),
                   "kt_mxfp4_moe_decode")
        else:
            _check(L.kt_moe_route_permute(logits.data_ptr(), T, self.E, self.k, self.renormalize, ids.data_ptr(),
                                          w.data_ptr(), offs.data_ptr(), perm.data_ptr(), inv.data_ptr(),
                                          rws.data_ptr(), rws.numel(), sp), "kt_moe_route_permute")
            _check(L.kt_mxfp4_moe_forward_routed(hidden.data_ptr(), T, self.H, ids.data_ptr(), w.data_ptr(), self.k,
                                                 offs.data_ptr(), perm.data_ptr(), inv.data_ptr(), w13, w13_sf, w2,
                                                 w2_sf, self.E, self.I, out.data_ptr(), ws.data_ptr(), ws.numel(),
                                                 self._optsref, sp), "kt_mxfp4_moe_forward_routed")


class Layerwise:
    """Layerwise prefill over L layers whose packed experts live in pinned host memory."""

    def __init__(self, host_packs: list[torch.Tensor], H: int, I: int, E: int, k: int, T_max: int,
                 zero_copy: bool = False):
        """zero_copy=False: two device slots, the next layer copied while the current one computes.
        zero_copy=True: the GEMMs read each layer's experts in place from the pinned host packs."""
        self.H, self.I, self.E, self.k, self.T_max = H, I, E, k, T_max
        self.zero_copy = bool(zero_copy)
        need = int(lib().kt_layerwise_pack_bytes(H, I, E))
        for p in host_packs:
            if p.device.type != "cpu" or not p.is_pinned() or p.dtype != torch.uint8 or p.numel() < need:
                raise ValueError(f"each host pack must be a pinned uint8 CPU tensor of >= {need} bytes")
        self._packs = list(host_packs)     # keep them alive
        self.L = len(host_packs)
        arr = (ctypes.c_void_p * len(host_packs))(*[p.data_ptr() for p in host_packs])
        h = ctypes.c_void_p()
        create = lib().kt_layerwise_create_zero_copy if self.zero_copy else lib().kt_layerwise_create
        _check(create(ctypes.byref(h), len(host_packs), H, I, E, k, T_max, arr), "kt_layerwise_create")
        self._h = h

    def enable_timing(self, enable: bool = True):
        """Record per-layer copy / compute events in the following prefills."""
        _check(lib().kt_layerwise_enable_timing(self._h, int(bool(enable))), "kt_layerwise_enable_timing")

    def timing(self) -> dict:
        """{"layers": [(copy_ms, compute_ms)] per layer, "span_ms": ...} of the most recent prefill."""
        cp = (ctypes.c_double * self.L)()
        cm = (ctypes.c_double * self.L)()
        span = ctypes.c_double()
        _check(lib().kt_layerwise_read_timing(self._h, cp, cm, ctypes.byref(span)), "kt_layerwise_read_timing")
        return {"layers": [(float(cp[i]), float(cm[i])) for i in range(self.L)], "span_ms": float(span.value)}

    @staticmethod
    def pack_bytes(H: int, I: int, E: int) -> int:
        return int(lib().kt_layerwise_pack_bytes(H, I, E))

    @staticmethod
    def pack_offsets(H: int, I: int, E: int) -> tuple[int, int, int, int]:
        o = [ctypes.c_size_t() for _ in range(4)]
        _check(lib().kt_layerwise_pack_offsets(H, I, E, *[ctypes.byref(x) for x in o]), "kt_layerwise_pack_offsets")
        return tuple(int(x.value) for x in o)

    @classmethod
    def pack(cls, w13, w13_sf, w2, w2_sf, out: torch.Tensor | None = None) -> torch.Tensor:
        """Pack one layer's weights into a pinned host buffer (w13 | w13_sf | w2 | w2_sf)."""
        E, I, H = check_fc_shapes(w13, w2)
        n = cls.pack_bytes(H, I, E)
        if out is None:
            out = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        offs = cls.pack_offsets(H, I, E)
        for off, t in zip(offs, (w13, w13_sf, w2, w2_sf)):
            out[off:off + t.numel()].copy_(t.reshape(-1), non_blocking=False)
        return out

    def inject_copy_failure(self, layer: int):
        _check(lib().kt_layerwise_inject_copy_failure(self._h, layer), "kt_layerwise_inject_copy_failure")

    def prefill(self, hidden: torch.Tensor, logits: list[torch.Tensor], out: torch.Tensor | None = None,
                serialized: bool = False, stream=None) -> torch.Tensor:
        _need(hidden, "hidden", torch.bfloat16, 2)
        dev = hidden.device
        T = hidden.shape[0]
        for lg in logits:
            _need(lg, "logits", torch.float32, 2, dev)
        if out is None:
            out = torch.empty_like(hidden)
        arr = (ctypes.c_void_p * len(logits))(*[lg.data_ptr() for lg in logits])
        with torch.cuda.device(dev):
            _check(lib().kt_layerwise_prefill(self._h, _ptr(hidden), arr, _ptr(out), T, int(bool(serialized)),
                                              _stream_ptr(stream, dev)), "kt_layerwise_prefill")
        return out

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _check(lib().kt_layerwise_destroy(self._h), "kt_layerwise_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass
