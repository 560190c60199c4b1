"""Host-side checks of the C ABI (no GPU needed).

The library must build and export every function include/kt_moe.h declares,
and every argument check must return its documented status before anything
touches the GPU.  Pointers here are fake, non-null addresses that are never
dereferenced: every case below fails a check first.
"""
import ctypes
import os
import re

import pytest
import torch

import mxfp4_weight_moe_gb300 as kt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kt_moe.h")

KT_OK, INVALID, SHAPE, WS, CUDA, TIMEOUT, DEVTIMEOUT, ALIGN, BADID = 0, -1, -2, -3, -4, -5, -6, -7, -8
P = 0x7F0000000000          # fake 1 KB-aligned device address (never dereferenced)


def declared_functions():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(kt_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("kt_moe_route_permute", "kt_mxfp4_moe_forward", "kt_moe_workspace_bytes",
                 "kt_moe_read_device_error", "kt_layerwise_create", "kt_layerwise_prefill", "kt_layerwise_destroy",
                 "kt_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol():
    L = kt.lib()
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    assert set(declared_functions()) <= set(kt._SIGNATURES), "binding lacks a declared entry point"


def test_status_strings():
    for code, name in ((KT_OK, "KT_OK"), (INVALID, "KT_ERR_INVALID_ARG"), (SHAPE, "KT_ERR_UNSUPPORTED_SHAPE"),
                       (WS, "KT_ERR_WORKSPACE"), (CUDA, "KT_ERR_CUDA"), (TIMEOUT, "KT_ERR_TIMEOUT"),
                       (DEVTIMEOUT, "KT_ERR_DEVICE_TIMEOUT"), (ALIGN, "KT_ERR_ALIGNMENT"),
                       (BADID, "KT_ERR_BAD_EXPERT_ID")):
        assert kt.status_string(code) == name


def _fwd(T=4, H=256, I=256, E=8, k=2, hidden=P, ids=P, w=P, w13=P, w13_sf=P, w2=P, w2_sf=P, out=P, ws=P,
         ws_bytes=None):
    L = kt.lib()
    if ws_bytes is None:
        ws_bytes = 0     # too small unless a test overrides it
    v = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.kt_mxfp4_moe_forward(v(hidden), T, H, v(ids), v(w), k, v(w13), v(w13_sf), v(w2), v(w2_sf), E, I,
                                  v(out), v(ws), ws_bytes, None)


def test_forward_shape_checks():
    assert _fwd(T=-1) == INVALID
    assert _fwd(E=0) == INVALID
    assert _fwd(k=0) == INVALID
    assert _fwd(k=9, E=8) == INVALID
    assert _fwd(E=1025, k=2) == SHAPE
    assert _fwd(E=64, k=33) == SHAPE
    assert _fwd(H=100) == SHAPE
    assert "multiples of 128" in kt.lib().kt_last_error().decode()
    assert _fwd(I=64) == SHAPE
    assert _fwd(H=0) == INVALID


def test_forward_zero_tokens_is_a_noop():
    # T == 0 returns before any pointer is looked at or any launch happens
    assert _fwd(T=0, hidden=None, ids=None, w=None, w13=None, w13_sf=None, w2=None, w2_sf=None, out=None,
                ws=None) == KT_OK


def test_forward_pointer_and_workspace_checks():
    assert _fwd(hidden=None) == INVALID
    assert _fwd(w2_sf=None) == INVALID
    assert _fwd(ws=None) == INVALID
    assert _fwd(hidden=P + 2) == ALIGN
    assert _fwd(out=P + 8) == ALIGN
    assert _fwd(w13=P + 16) == ALIGN          # fp4 weights need 32 bytes
    assert _fwd(w2_sf=P + 4) == ALIGN
    need = kt.workspace_bytes(4, 256, 256, 8, 2)
    assert need > 0
    assert _fwd(ws=P + 128, ws_bytes=need) == WS      # not 256-byte aligned
    assert _fwd(ws_bytes=need - 1) == WS
    assert "workspace" in kt.lib().kt_last_error().decode()


def test_routed_forward_checks():
    """kt_mxfp4_moe_forward_routed: the forward's checks, then its own routing arrays (null, alignment)."""
    L = kt.lib()
    v = lambda x: None if x is None else ctypes.c_void_p(x)

    def fwd(off=P, perm=P, inv=P, T=4, H=256, I=256, E=8, k=2, hidden=P, ws_bytes=0):
        return L.kt_mxfp4_moe_forward_routed(v(hidden), T, H, v(P), v(P), k, v(off), v(perm), v(inv), v(P), v(P),
                                             v(P), v(P), E, I, v(P), v(P), ws_bytes, None, None)

    assert fwd(T=-1) == INVALID
    assert fwd(H=100) == SHAPE
    assert fwd(T=0, off=None, perm=None, inv=None) == KT_OK
    assert fwd(off=None) == INVALID
    assert fwd(inv=None) == INVALID
    assert "routing" in L.kt_last_error().decode()
    assert fwd(hidden=None, off=None) == INVALID
    assert fwd(perm=P + 4) == ALIGN
    need = kt.workspace_bytes(4, 256, 256, 8, 2)
    assert fwd(ws_bytes=need - 1) == WS


def _route(T=4, E=8, k=2, logits=P, ids=P, w=P, off=P, perm=P, inv=P, ws=P, ws_bytes=0):
    v = lambda x: None if x is None else ctypes.c_void_p(x)
    return kt.lib().kt_moe_route_permute(v(logits), T, E, k, 1, v(ids), v(w), v(off), v(perm), v(inv), v(ws),
                                         ws_bytes, None)


def test_route_checks():
    assert _route(T=-3) == INVALID
    assert _route(k=9) == INVALID
    assert _route(E=2048) == SHAPE
    assert _route(T=0, logits=None) == KT_OK
    assert _route(logits=None) == INVALID
    assert _route(perm=P + 2) == ALIGN
    need = kt.lib().kt_moe_route_workspace_bytes(4, 8, 2)
    assert need > 0
    assert _route(ws_bytes=need - 1) == WS
    assert _route(ws=P + 64, ws_bytes=need) == WS


def test_grouped_gemm_checks():
    L = kt.lib()
    v = ctypes.c_void_p
    assert L.kt_mx_grouped_gemm_f32(v(P), v(P), 10, 100, v(P), v(P), v(P), 2, 128, v(P), v(P), 1 << 20, None) == SHAPE
    assert L.kt_mx_grouped_gemm_f32(v(P), v(P), 10, 128, v(P), v(P), v(P), 2, 96, v(P), v(P), 1 << 20, None) == SHAPE
    assert L.kt_mx_grouped_gemm_f32(None, v(P), 10, 128, v(P), v(P), v(P), 2, 128, v(P), v(P), 1 << 20, None) == INVALID
    assert L.kt_mx_grouped_gemm_f32(v(P), v(P), 10, 128, v(P), v(P + 16), v(P), 2, 128, v(P), v(P), 1 << 20,
                                    None) == ALIGN
    assert L.kt_mx_grouped_gemm_f32(v(P), v(P), 10, 128, v(P), v(P), v(P), 2, 128, v(P), v(P), 8, None) == WS
    assert L.kt_mx_gemm_workspace_bytes(10, 128, 2) > 1024
    assert L.kt_mx_grouped_gemm_f32(v(P), v(P), 0, 128, None, None, None, 2, 128, None, None, 0, None) == KT_OK


def test_kstep_major_scale_view_roundtrip():
    S, K = 7, 512
    plain = torch.randint(0, 255, (S, K // 32), dtype=torch.uint8)
    S4 = 8
    words = torch.zeros(K // 128, S4, 4, dtype=torch.uint8)
    for r in range(S):
        for b in range(K // 32):
            words[b // 4, r, b % 4] = plain[r, b]
    assert torch.equal(kt.scales_from_kstep_major(words.reshape(-1), S, K), plain)


def test_workspace_layout_is_ordered_and_aligned():
    T, H, I, E, k = 4096, 4096, 2048, 256, 6
    lay = kt.workspace_layout(T, H, I, E, k)
    S = T * k
    order = ["err", "expert_offsets", "chunk_prefix", "perm", "inv_perm", "hist", "a1", "a1_sf", "a2", "a2_sf", "y",
             "total"]
    offs = [lay[n] for n in order]
    assert offs == sorted(offs) and all(o % 1024 == 0 for o in offs)
    assert lay["a1_sf"] - lay["a1"] >= S * H
    assert lay["a2_sf"] - lay["a2"] >= S * I
    assert lay["total"] - lay["y"] >= S * H * 2
    assert kt.workspace_bytes(T, H, I, E, k) == lay["total"]
    assert kt.workspace_bytes(T, 100, I, E, k) == 0


def test_layerwise_checks_and_pack_layout():
    L = kt.lib()
    H, I, E = 4096, 2048, 256
    offs = kt.Layerwise.pack_offsets(H, I, E)
    sizes = [E * 2 * I * H // 2, E * 2 * I * H // 32, E * H * I // 2, E * H * I // 32]
    assert offs[0] == 0
    for a, b, s in zip(offs, list(offs[1:]) + [kt.Layerwise.pack_bytes(H, I, E)], sizes):
        assert b - a >= s and a % 256 == 0
    assert kt.Layerwise.pack_bytes(H, I, E) == pytest.approx(3.4226e9, rel=1e-3)
    h = ctypes.c_void_p()
    packs = (ctypes.c_void_p * 2)(P, P)
    assert L.kt_layerwise_create(None, 2, H, I, E, 6, 16, packs) == INVALID
    assert L.kt_layerwise_create(ctypes.byref(h), 2, 100, I, E, 6, 16, packs) == SHAPE
    assert L.kt_layerwise_create(ctypes.byref(h), 0, H, I, E, 6, 16, packs) == INVALID
    assert L.kt_layerwise_prefill(None, None, None, None, 1, 0, None) == INVALID
    assert L.kt_layerwise_destroy(None) == INVALID


def test_python_wrapper_checks_fc1_is_twice_fc2():
    # official test shape: fc1 inter 256 = 2 x fc2 inter 128 is the gated layout
    w13 = torch.zeros(2, 256, 64, dtype=torch.uint8)
    w2 = torch.zeros(2, 128, 64, dtype=torch.uint8)
    assert kt.check_fc_shapes(w13, w2) == (2, 128, 128)
    with pytest.raises(ValueError, match="256"):
        kt.check_fc_shapes(torch.zeros(2, 128, 64, dtype=torch.uint8), w2)


def test_moe_layer_rejects_cpu_weights():
    E, H, I = 2, 128, 128
    W = (torch.zeros(E, 2 * I, H // 2, dtype=torch.uint8), torch.zeros(E, 2 * I, H // 32, dtype=torch.uint8),
         torch.zeros(E, H, I // 2, dtype=torch.uint8), torch.zeros(E, H, I // 32, dtype=torch.uint8))
    with pytest.raises(ValueError):
        kt.MoeLayer(*W, 2)


def test_ops_reject_cpu_tensors():
    x = torch.zeros(2, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        kt.forward(x, torch.zeros(2, 1, dtype=torch.int32), torch.zeros(2, 1), torch.zeros(1, 512, 128, dtype=torch.uint8),
                   torch.zeros(1, 512, 8, dtype=torch.uint8), torch.zeros(1, 256, 128, dtype=torch.uint8),
                   torch.zeros(1, 256, 8, dtype=torch.uint8))


def test_debug_configure_rejects_unknown_flags():
    with pytest.raises(kt.KTError):
        kt.debug_configure(0, 0x80)
    kt.debug_configure()


def test_profile_stage_mask_rejects_unknown_stages():
    assert kt.lib().kt_moe_profile_enable_stages(1 << len(kt.STAGES)) == -1   # KT_ERR_INVALID_ARG
    assert kt.lib().kt_moe_profile_enable_stages(0) == 0


def _kernel_bodies(src: str) -> dict:
    """name -> body text of every __global__ function in a CUDA source."""
    import re
    out = {}
    for m in re.finditer(r"__global__\s+void\s+(?:__launch_bounds__\([^)]*\)\s*)?(\w+)\s*\(", src):
        start = src.index("{", m.end())
        depth, i = 0, start
        while True:
            if src[i] == "{":
                depth += 1
            elif src[i] == "}":
                depth -= 1
                if depth == 0:
                    break
            i += 1
        out[m.group(1)] = src[start:i + 1]
    return out


def test_chained_kernels_wait_before_touching_memory():
    """Kernels launched with programmatic stream serialization may start while
    their predecessor runs; each must call griddep_wait() before its first
    global-memory access (checked here as: before any pointer argument is
    read through __ldg, an index or a dereference of a kernel parameter)."""
    import glob
    import os
    import re
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "mxfp4_weight_moe_gb300", "csrc")
    src = "\n".join(open(f).read() for f in sorted(glob.glob(os.path.join(csrc, "*.cu"))))
    # launch_chained(<kernel>, ...) calls, and the routing launcher's go(route_topk_kernel<EPL>)
    chained = (set(re.findall(r"launch_chained\((\w+)", src)) - {"kernel"}) | set(re.findall(r"go\((\w+)<", src))
    assert "cudaLaunchAttributeProgrammaticStreamSerialization" in src
    chained.add("mx_gemm_kernel")   # launched with the attribute through cudaLaunchKernelEx
    bodies = _kernel_bodies(src)
    assert chained <= set(bodies), chained - set(bodies)
    # the GEMM kernels delegate to gemm_body (shared with the single-launch decode kernel)
    assert "gemm_body<MODE, 1, NEAR>" in bodies["mx_gemm_kernel"]
    m = re.search(r"void\s+gemm_body\s*\(", src)
    start = src.index("{", m.end())
    depth, i = 0, start
    while True:
        depth += {"{": 1, "}": -1}.get(src[i], 0)
        if depth == 0:
            break
        i += 1
    bodies["mx_gemm_kernel"] = src[start:i + 1]
    for name in sorted(chained):
        body = bodies[name]
        assert "griddep_wait();" in body, name
        before = body[:body.index("griddep_wait();")]
        assert "__ldg(" not in before and not re.search(r"\bp\.\w+\s*\[", before), name
