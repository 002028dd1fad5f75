"""The global gradient norm computed while the optimiser step folds the deferred gradient
partials (each fold also sums the squares of the final values it writes; only the gradient
ranges no fold finalises, such as wte and wpe, are read again) equals the norm of the
gradients read back, and the clipped AdamW step that uses it equals the one that uses the
norm from a full pass over the gradients (the clip of the 124M optimiser step,
min(1, c / (||g|| + 1e-6)); AdamW of 「从零实现一个最小GPT」 三.9)."""
import numpy as np
import pytest
import torch

from decoder_only_transformer_05_b300 import synthetic as S

pytestmark = pytest.mark.gpu

G = None


@pytest.fixture(scope="module", autouse=True)
def lib():
    global G
    from decoder_only_transformer_05_b300 import build, gpt2
    build.build()
    gpt2.load_library()
    G = gpt2
    yield


def step(name, B, read_grads_first):
    w = S.WORKLOADS[name]
    m = G.GPT2(vocab_size=w["V"], padded_vocab_size=w["Vp"], block_size=w["T"],
               n_layer=w["L"], n_head=w["H"], n_embd=w["C"], batch_size=B, bias=w["bias"],
               precision=w["precision"], init=False)
    params = S.init_params(w["w_seed"], w["V"], w["Vp"], w["T"], w["L"], w["C"], w["bias"])
    m.set_params(params)
    m.zero_grad()
    for i in range(3):
        tok, tgt = S.batch(w["tok_seed"], 60 + i, B, w["T"], w["V"], w["dist"], w["s"])
        m.forward_backward(torch.tensor(tok).cuda(), torch.tensor(tgt).cuda(), B, w["T"], 1 / 3)
    flat = m.read_region("grads", np.float32) if read_grads_first else None
    norm = m.adamw_step(1e-3, 0.9, 0.95, 1e-8, 0.1, grad_clip=1.0, want_norm=True)
    p = m.read_region("params", np.float32)
    m.close()
    return norm, p, flat


@pytest.mark.parametrize("name,B", [("char-bf16", 8), ("tiny-fp32", 4)])
def test_norm_from_the_folds_matches_a_full_pass(name, B):
    n_fold, p_fold, _ = step(name, B, False)        # the step folds: fold-time norm
    n_full, p_full, g = step(name, B, True)         # folded earlier: full pass
    ref = float(np.sqrt((g.astype(np.float64) ** 2).sum()))
    assert abs(n_full - ref) / ref <= 1e-5
    assert abs(n_fold - ref) / ref <= 1e-5
    assert n_fold > 1.0                             # the clip is active (coefficient < 1)
    assert np.abs(p_fold - p_full).max() <= 1e-6 * max(np.abs(p_full).max(), 1.0)
