"""GPU: the prefill-shaped configurations at full size (DeepSeek-V4-Flash-
shaped T=4096; Kimi-K3-shaped T=16 and T=8192), same launch path as the
benchmark.  Routing and permutation are checked in full; outputs, A1 and A2
on a stratified token sample (each token's output depends only on its own
row and routing, so a sample is exact, not approximate)."""
import numpy as np
import pytest
import torch

import oracle as O
from mxfp4_weight_moe_gb300 import synthetic as syn

from helpers import sample_tokens
from test_gpu_3_forward import _check_case

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.mark.parametrize("name,n_sample", [("dsv4", 256), ("kimi_T16", 16), ("kimi_T8192", 64)])
def test_full_size_config(name, n_sample):
    cfg = syn.CONFIGS[name]
    hidden = syn.make_hidden(cfg.T, cfg.H, cfg.seed, device="cuda")
    logits = syn.make_logits(cfg.T, cfg.E, cfg.logits, cfg.seed, device="cuda")
    ids, w = O.route(logits.cpu().numpy(), cfg.k)
    W = syn.make_weights(cfg.E, cfg.H, cfg.I, seed=cfg.seed, device="cuda")
    tokens = sample_tokens(ids, n_sample, seed=1)
    _check_case(hidden, ids, w, W, tokens=tokens)
    del W
    torch.cuda.empty_cache()
