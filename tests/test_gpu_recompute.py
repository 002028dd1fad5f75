"""Activation recomputation (gpt2_config.recompute = 1): the backward recomputes both
LayerNorm outputs of each layer and the MLP's gelu(u), gelu'(u) from the kept
pre-activation instead of keeping them, which frees 2 [B*T, C] + [B*T, 4C] activation
elements per layer. The forward is the same computation, so its loss is bit-identical to
the ordinary handle's; the gradients differ only by the rounding of u to bf16, and both
are held to the bf16 parity bounds against the oracle (loss within 2e-2, gradient cosine
>= 0.999; 「从零实现一个最小GPT」 三.7 and 三.9)."""
import numpy as np
import pytest
import torch

from decoder_only_transformer_05_b300 import synthetic as S
from oracle import gpt2_oracle as O

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


def cosine(a, r):
    a, r = np.asarray(a, np.float64).reshape(-1), np.asarray(r, np.float64).reshape(-1)
    return float(a @ r / (np.linalg.norm(a) * np.linalg.norm(r) + 1e-300))


def run(name, B, recompute, precision=None, graph=None):
    w = S.WORKLOADS[name]
    m = G.GPT2(vocab_size=w["V"], padded_vocab_size=w["Vp"], block_size=w["T"],
               n_layer=w["L"], n_head=w["H"], n_embd=w["C"], batch_size=B, bias=w["bias"],
               precision=precision or w["precision"], init=False, recompute=recompute)
    params = S.init_params(w["w_seed"], w["V"], w["Vp"], w["T"], w["L"], w["C"], w["bias"])
    m.set_params(params)
    tok, tgt = S.batch(w["tok_seed"], 4, B, w["T"], w["V"], w["dist"], w["s"])
    dtok, dtgt = torch.tensor(tok).cuda(), torch.tensor(tgt).cuda()
    m.zero_grad()
    if graph is not None:   # two micro-batches, recorded as a CUDA graph and replayed, or eager
        m.set_graph_mode(graph)
        m.forward_backward(dtok, dtgt, B, w["T"], 0.5)
        m.forward_backward(dtok, dtgt, B, w["T"], 0.5)
        loss = m.get_loss()
    else:
        loss = m.forward(dtok, dtgt, want_loss=True)
        m.backward(1.0)
    grads = m.get_grads()
    mem = m.memory_bytes()
    m.close()
    return loss, grads, mem, params, tok, tgt, w


@pytest.mark.parametrize("name,B", [("char-bf16", 8), ("gpt2-124m-micro", 1)])
def test_recompute_matches_oracle_and_saves_memory(name, B):
    loss0, g0, mem0, params, tok, tgt, w = run(name, B, False)
    loss1, g1, mem1, _, _, _, _ = run(name, B, True)
    assert loss1 == loss0                      # the forward is unchanged
    M, C, L = B * w["T"], w["C"], w["L"]
    saved = mem0[1] - mem1[1]
    want = L * (2 * M * C + 4 * M * C) * 2 - (M * C + 4 * M * C) * 2   # less the shared buffers
    assert saved >= want, (saved, want)
    cfg = O.Config(w["V"], w["Vp"], w["T"], w["L"], w["H"], w["C"], w["bias"])
    ref = O.forward(params, cfg, tok, tgt)
    rg = O.backward(params, cfg, ref["cache"], 1.0)
    assert abs(loss1 - ref["loss"]) <= 2e-2
    cos = {k: cosine(g1[k], rg[k]) for k in g1}
    assert min(cos.values()) >= 0.999, cos
    near = {k: cosine(g1[k], g0[k]) for k in g1}
    assert min(near.values()) >= 0.9999, near


def test_recompute_fp32_and_graph_replay():
    # fp32 path: the recomputation is exact up to fp32 rounding of the same operations
    loss0, g0, _, params, tok, tgt, w = run("tiny-fp32", 4, False)
    loss1, g1, _, _, _, _, _ = run("tiny-fp32", 4, True)
    assert loss1 == loss0
    for k in g0:
        assert np.abs(g1[k] - g0[k]).max() <= 1e-5 * max(np.abs(g0[k]).max(), 1e-30), k
    # bf16 with the micro-batch recorded as a CUDA graph and replayed
    lg, gg, _, _, _, _, _ = run("char-bf16", 4, True, graph=True)
    le, ge, _, _, _, _, _ = run("char-bf16", 4, True, graph=False)
    assert lg == le
    for k in ge:
        assert np.array_equal(gg[k], ge[k]), k
