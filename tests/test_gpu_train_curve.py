"""The char-level configuration trained for 100 optimiser steps on the GPU beside the CPU
oracle: per-step losses of the two runs, from the same initial weights and the same seeded
batches, with AdamW and the cosine learning-rate schedule 1e-3 -> 1e-4 (the shrunken
reproduction of 「4.1 GPT-2 (124M) 复现」 section 3.4, AdamW of 「从零实现一个最小GPT」
section 三.9, clip 1.0).

The bf16 run drifts from the float64 one as the steps compound, so this is a band, not a
parity gate: every step within 0.1 of the oracle's loss (five times the one-step bf16
bound of 2e-2), and the last 20 steps within 0.05 on average. The batch is reduced to two
sequences so the oracle's 100 steps take a few minutes.
"""
import numpy as np
import pytest
import torch

from decoder_only_transformer_05_b300 import synthetic as S
from oracle import gpt2_oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def lib():
    from decoder_only_transformer_05_b300 import build, gpt2
    build.build()
    gpt2.load_library()
    yield


def test_char_model_100_steps_tracks_the_oracle():
    from decoder_only_transformer_05_b300 import gpt2 as G
    w = S.WORKLOADS["char-bf16"]
    B, steps = 2, 100
    m = G.GPT2(vocab_size=w["V"], padded_vocab_size=w["Vp"], block_size=w["T"],
               n_layer=w["L"], n_head=w["H"], n_embd=w["C"], batch_size=B, bias=w["bias"],
               precision="bf16", init=False)
    params = S.init_params(w["w_seed"], w["V"], w["Vp"], w["T"], w["L"], w["C"], w["bias"])
    m.set_params(params)
    cfg = O.Config(w["V"], w["Vp"], w["T"], w["L"], w["H"], w["C"], w["bias"])
    batches = [S.batch(w["tok_seed"], 100 + it, B, w["T"], w["V"], w["dist"], w["s"])
               for it in range(steps)]

    gpu = []
    for it, (tok, tgt) in enumerate(batches):
        m.zero_grad()
        m.forward_backward(torch.tensor(tok).cuda(), torch.tensor(tgt).cuda(), B, w["T"], 1.0)
        gpu.append(m.get_loss())
        m.adamw_step(O.lr_cosine(it), 0.9, 0.95, 1e-8, 0.1, grad_clip=1.0)
    m.close()

    p = {k: np.asarray(v, np.float64) for k, v in params.items()}
    mo = {k: np.zeros_like(v) for k, v in p.items()}
    vo = {k: np.zeros_like(v) for k, v in p.items()}
    ref = []
    for it, mb in enumerate(batches):
        p, mo, vo, loss, _, _ = O.training_step(p, mo, vo, it + 1, cfg, [mb], O.lr_cosine(it),
                                                0.9, 0.95, 1e-8, 0.1, 1.0)
        ref.append(loss)

    gpu, ref = np.array(gpu), np.array(ref)
    diff = np.abs(gpu - ref)
    print("\nstep  gpu     oracle")
    for it in range(0, steps, 10):
        print(f"{it:4d}  {gpu[it]:.4f}  {ref[it]:.4f}")
    print(f"max |diff| {diff.max():.4f}, mean of the last 20 {diff[-20:].mean():.4f}")
    assert abs(gpu[0] - ref[0]) <= 2e-2
    assert diff.max() <= 0.1
    assert diff[-20:].mean() <= 0.05
    assert ref[-20:].mean() < ref[:5].mean()       # the run does learn
