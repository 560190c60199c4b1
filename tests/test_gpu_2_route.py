"""GPU: routing and permutation must equal the oracle bit for bit (ids,
expert offsets, perm, inv_perm); gating weights within 2 f32 ulp (both
sides compute them in fp64 and round once)."""
import numpy as np
import pytest
import torch

import mxfp4_weight_moe_gb300 as kt
import oracle as O
from mxfp4_weight_moe_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _check(logits: torch.Tensor, k: int, renorm: bool = True):
    ids, w, off, perm, inv = kt.route_permute(logits, k, renormalize=renorm)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    rid, rw = O.route(lg, k, renorm)
    roff, rperm, rinv, bad = O.permute(rid, lg.shape[1])
    assert bad == 0
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_array_equal(off.cpu().numpy(), roff)
    np.testing.assert_array_equal(perm.cpu().numpy(), rperm)
    np.testing.assert_array_equal(inv.cpu().numpy(), rinv)
    gw = w.cpu().numpy().astype(np.float64)
    ulp = np.spacing(np.abs(rw)).astype(np.float64)
    assert np.all(np.abs(gw - rw) <= 2 * ulp), float((np.abs(gw - rw) / ulp).max())
    return rid


@pytest.mark.parametrize("name", ["tiny", "small_T1", "small_T2", "small_T8", "small_T32", "dsv4", "kimi_T16",
                                  "kimi_T8192"])
def test_route_configs(name):
    cfg = syn.CONFIGS[name]
    logits = syn.make_logits(cfg.T, cfg.E, cfg.logits, seed=cfg.seed, device="cuda")
    rid = _check(logits, cfg.k)
    if name.startswith("small"):
        counts = np.bincount(rid.reshape(-1), minlength=cfg.E)
        assert counts[0] == cfg.T and counts[cfg.E - 1] == 0


@pytest.mark.parametrize("renorm", [True, False])
def test_route_ties_and_modes(renorm):
    g = torch.Generator(device="cuda").manual_seed(3)
    logits = torch.randn(300, 40, generator=g, device="cuda")
    logits[0] = 0.25                  # all tied
    logits[1, 5] = logits[1, 9] = 7.0
    logits[2, :] = torch.arange(40, device="cuda").float() * 0   # zeros
    _check(logits, 7, renorm)


def test_route_k_equals_E_and_ragged_tiles():
    g = torch.Generator(device="cuda").manual_seed(4)
    _check(torch.randn(1, 2, generator=g, device="cuda"), 2)
    _check(torch.randn(777, 32, generator=g, device="cuda"), 32)     # k = E = 32, slots not a tile multiple
    _check(torch.randn(5000, 1024, generator=g, device="cuda"), 32)  # largest E and k supported
