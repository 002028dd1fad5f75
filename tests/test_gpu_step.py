"""Whole training-step parity on the GPU, through the C ABI (include/gpt2.h), against the
float64 CPU oracle on identical seeded inputs and weights.

Gates:
  fp32 path: loss relative error <= 1e-5, every gradient tensor <= 1e-3 infinity-norm
  relative error, every updated parameter tensor <= 1e-3 (AdamW checked on the GPU's own
  gradients, and end to end away from near-zero gradients, where m/sqrt(v) ~ sign(g)
  amplifies any gradient error), embedding gather bit-exact.
  bf16 path: |loss - loss_ref| <= 2e-2, cosine similarity >= 0.999 per gradient tensor.
"""
import math

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


def make(name, B=None, init_seed=None):
    w = S.WORKLOADS[name]
    B = B or w["B"]
    m = G.GPT2(vocab_size=w["V"], padded_vocab_size=w["Vp"], block_size=w["T"],
               n_layer=w["L"], n_head=w["H"], n_embd=w["C"], batch_size=B, bias=w["bias"],
               precision=w["precision"], init=False)
    params = S.init_params(w["w_seed"] if init_seed is None else init_seed, w["V"], w["Vp"],
                           w["T"], w["L"], w["C"], w["bias"])
    m.set_params(params)
    cfg = O.Config(w["V"], w["Vp"], w["T"], w["L"], w["H"], w["C"], w["bias"])
    return m, params, cfg, w


def tokens_for(w, B, index=0):
    tok, tgt = S.batch(w["tok_seed"], index, B, w["T"], w["V"], w["dist"], w["s"])
    return tok, tgt, torch.tensor(tok).cuda(), torch.tensor(tgt).cuda()


def rel_inf(a, r):
    return float(np.abs(a - r).max() / max(np.abs(r).max(), 1e-30))


def cosine(a, r):
    a, r = np.asarray(a, np.float64).reshape(-1), np.asarray(r, np.float64).reshape(-1)
    return float(a @ r / (np.linalg.norm(a) * np.linalg.norm(r) + 1e-300))


# ----------------------------------------------------------------- fp32 path
@pytest.fixture(scope="module")
def tiny():
    m, params, cfg, w = make("tiny-fp32")
    tok, tgt, dtok, dtgt = tokens_for(w, w["B"])
    loss = m.forward(dtok, dtgt, want_loss=True)
    x0 = m.read_region("encoded", np.float32, count=w["B"] * w["T"] * w["C"])
    losses = m.read_region("losses", np.float32, count=w["B"] * w["T"])
    m.zero_grad()
    m.backward(1.0)
    grads = m.get_grads()
    ref = O.forward(params, cfg, tok, tgt)
    rgrads = O.backward(params, cfg, ref["cache"], 1.0)
    return dict(m=m, params=params, cfg=cfg, w=w, tok=tok, tgt=tgt, dtok=dtok, dtgt=dtgt,
                loss=loss, x0=x0, losses=losses, grads=grads, ref=ref, rgrads=rgrads)


def test_fp32_loss(tiny):
    ref = tiny["ref"]["loss"]
    assert abs(tiny["loss"] - ref) / ref <= 1e-5
    np.testing.assert_allclose(tiny["losses"], tiny["ref"]["losses"].reshape(-1), rtol=1e-5,
                               atol=1e-6)


def test_fp32_embedding_gather_is_bit_exact(tiny):
    p, tok, w = tiny["params"], tiny["tok"], tiny["w"]
    expect = (p["wte"][tok] + p["wpe"][None, :w["T"]]).astype(np.float32).reshape(-1)
    assert np.array_equal(tiny["x0"], expect)


def test_fp32_gradients(tiny):
    for name, g in tiny["grads"].items():
        r = tiny["rgrads"][name]
        assert rel_inf(g, r) <= 1e-3, (name, rel_inf(g, r))


def test_fp32_gradients_with_linear_biases():
    # the tiny model with biases on every Linear layer (non-zero, so the forward adds
    # them too): the projection biases' gradients come from the LayerNorm backward's
    # column sums, the fc/qkv ones from the column-sum kernel
    w = dict(S.WORKLOADS["tiny-fp32"])
    w["bias"] = True
    m = G.GPT2(vocab_size=w["V"], padded_vocab_size=w["Vp"], block_size=w["T"],
               n_layer=w["L"], n_head=w["H"], n_embd=w["C"], batch_size=w["B"], bias=True,
               precision="fp32", init=False)
    params = S.init_params(w["w_seed"], w["V"], w["Vp"], w["T"], w["L"], w["C"], True)
    rng = np.random.default_rng(7)
    for k in ("qkvb", "attprojb", "fcb", "fcprojb"):
        params[k] = (0.02 * rng.standard_normal(params[k].shape)).astype(np.float32)
    m.set_params(params)
    tok, tgt, dtok, dtgt = tokens_for(w, w["B"])
    loss = m.forward(dtok, dtgt, want_loss=True)
    m.zero_grad()
    m.backward(1.0)
    grads = m.get_grads()
    cfg = O.Config(w["V"], w["Vp"], w["T"], w["L"], w["H"], w["C"], True)
    ref = O.forward(params, cfg, tok, tgt)
    rgrads = O.backward(params, cfg, ref["cache"], 1.0)
    assert abs(loss - ref["loss"]) / ref["loss"] <= 1e-5
    for name, g in grads.items():
        assert rel_inf(g, rgrads[name]) <= 1e-3, (name, rel_inf(g, rgrads[name]))
    m.close()


def test_fp32_adamw_update(tiny):
    m, params = tiny["m"], tiny["params"]
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.95, 1e-8, 0.1
    norm = m.adamw_step(lr, b1, b2, eps, wd, grad_clip=0.0, want_norm=True)
    new = m.get_params()
    gm, gv = m.get_moments()
    assert abs(norm - O.global_norm(tiny["rgrads"])) / norm < 1e-4
    zero = {k: np.zeros_like(v) for k, v in params.items()}
    for name in params:
        # (i) AdamW on the GPU's own gradients
        p1, m1, v1 = O.adamw_update(params[name], tiny["grads"][name], zero[name], zero[name], 1,
                                    lr, b1, b2, eps, wd)
        assert rel_inf(new[name], p1) <= 1e-3, name
        np.testing.assert_allclose(gm[name], m1, rtol=1e-5, atol=1e-12)
        np.testing.assert_allclose(gv[name], v1, rtol=1e-5, atol=1e-18)
        # (ii) end to end against the oracle's gradients, away from |g| ~ gradient error
        rg = tiny["rgrads"][name]
        p2, _, _ = O.adamw_update(params[name], rg, zero[name], zero[name], 1, lr, b1, b2, eps,
                                  wd)
        gerr = np.abs(tiny["grads"][name] - rg).max()
        keep = np.abs(rg) >= 1e3 * max(gerr, 1e-30)
        if keep.any():
            assert rel_inf(new[name][keep], p2[keep]) <= 1e-3, name
    m.step = 0


def test_fp32_gradient_accumulation_is_linear(tiny):
    m = tiny["m"]
    m.set_params(tiny["params"])      # the AdamW test moved them
    m.zero_grad()
    m.forward(tiny["dtok"], tiny["dtgt"])
    m.backward(0.5)
    m.forward(tiny["dtok"], tiny["dtgt"])
    m.backward(0.5)
    g2 = m.get_grads()
    for name in g2:
        if name == "wte":
            # the tied embedding gets two contributions per backward (lm_head and the
            # embedding scatter), so the fp32 rounding order of the sums differs; where
            # the two contributions cancel, an element's own relative error is unbounded,
            # so the bound is a few fp32 ulps of the tensor's largest element
            ref = tiny["grads"][name]
            ulp = np.float32(2.0 ** -24) * np.abs(ref).max()
            assert np.abs(g2[name] - ref).max() <= 8 * ulp, name
        else:
            assert np.array_equal(g2[name], tiny["grads"][name]), name


# ----------------------------------------------------------------- bf16 path
def bf16_step_check(name, B, loss_tol=2e-2, cos_min=0.999):
    m, params, cfg, w = make(name, B=B)
    tok, tgt, dtok, dtgt = tokens_for(w, B)
    loss = m.forward(dtok, dtgt, want_loss=True)
    m.zero_grad()
    m.backward(1.0)
    grads = m.get_grads()
    ref = O.forward(params, cfg, tok, tgt)
    rgrads = O.backward(params, cfg, ref["cache"], 1.0)
    assert abs(loss - ref["loss"]) <= loss_tol, (loss, ref["loss"])
    worst = {}
    for k in grads:
        worst[k] = cosine(grads[k], rgrads[k])
    bad = {k: v for k, v in worst.items() if v < cos_min}
    print(f"\n{name} B={B}: loss {loss:.6f} oracle {ref['loss']:.6f}; min grad cosine "
          f"{min(worst.values()):.6f} ({min(worst, key=worst.get)})")
    assert not bad, bad
    m.close()
    return loss, ref["loss"], worst


def test_bf16_char_model_full_batch():
    bf16_step_check("char-bf16", B=64)


def test_bf16_gpt2_124m_one_sequence():
    """The 124M shape (T = 1024, V = 50257 padded to 50304) on one sequence: the oracle
    computes the same per-row math as the full batch."""
    bf16_step_check("gpt2-124m-micro", B=1)


def test_bf16_gpt2_350m_shape_one_sequence():
    """The 350M shape (L = 24, H = 16, C = 1024, T = 1024) on one sequence against the
    oracle: loss and every gradient tensor."""
    bf16_step_check("gpt2-350m-shape", B=1)


def test_bf16_gpt2_124m_full_batch_sampled_rows():
    """At the full micro-batch (B = 12, as timed by the benchmark), per-position losses of
    sampled rows against the oracle run on those rows alone."""
    m, params, cfg, w = make("gpt2-124m-micro")
    B, T = w["B"], w["T"]
    tok, tgt, dtok, dtgt = tokens_for(w, B, index=3)
    loss = m.forward(dtok, dtgt, want_loss=True)
    losses = m.read_region("losses", np.float32, count=B * T).reshape(B, T)
    for b in (0, B - 1):
        ref = O.forward(params, cfg, tok[b:b + 1], tgt[b:b + 1])
        assert np.abs(losses[b] - ref["losses"][0]).max() < 5e-2
        assert abs(losses[b].mean() - ref["loss"]) < 1e-2
    assert abs(loss - losses.mean()) < 1e-4
    m.close()


def test_bf16_deterministic():
    m, params, cfg, w = make("char-bf16", B=8)
    tok, tgt, dtok, dtgt = tokens_for(w, 8)
    outs = []
    for _ in range(2):
        m.zero_grad()
        m.forward(dtok, dtgt)
        m.backward(1.0)
        outs.append(m.read_region("grads", np.float32))
    assert np.array_equal(outs[0], outs[1])
    m.close()


def test_forward_backward_graph_replay_matches_eager():
    """gpt2_forward_backward records the micro-batch as a CUDA graph on its first call and
    replays it afterwards: losses and accumulated gradients equal those of separate
    forward/backward calls bit for bit, for device and pinned-host token buffers."""
    m, params, cfg, w = make("char-bf16", B=8)
    batches = [tokens_for(w, 8, index=i) for i in range(4)]

    def run(use_fb, graph=True):
        m.set_params(params)
        m.set_graph_mode(graph)
        m.zero_grad()
        losses = []
        for i, (tok, tgt, dtok, dtgt) in enumerate(batches):
            if use_fb:
                if i % 2:   # pinned host buffers, copied in by the library
                    ht = torch.from_numpy(np.ascontiguousarray(tok)).pin_memory()
                    hg = torch.from_numpy(np.ascontiguousarray(tgt)).pin_memory()
                    m.forward_backward(ht, hg, 8, w["T"], 0.25)
                else:
                    m.forward_backward(dtok, dtgt, 8, w["T"], 0.25)
            else:
                m.forward(dtok, dtgt)
                m.backward(0.25)
            losses.append(m.get_loss())
        return losses, m.read_region("grads", np.float32)

    l_eager, g_eager = run(False)
    l_graph, g_graph = run(True)
    l_off, g_off = run(True, graph=False)
    assert len(set(l_eager)) == len(l_eager)     # the batches differ
    assert l_graph == l_eager and l_off == l_eager
    assert np.array_equal(g_graph, g_eager) and np.array_equal(g_off, g_eager)
    # profiling forces the eager path (events between launches); results unchanged
    m.set_graph_mode(True)
    m.profile_enable(("gemm",), capacity=4096)
    l_prof, g_prof = run(True)
    n, ms, flops = m.profile_read("gemm", reset=True)
    m.profile_enable((), capacity=0)
    assert n > 0 and l_prof == l_eager and np.array_equal(g_prof, g_eager)
    m.close()


def test_forward_backward_rejects_bad_shapes():
    m, params, cfg, w = make("char-bf16", B=8)
    tok, tgt, dtok, dtgt = tokens_for(w, 8)
    with pytest.raises(G.GPT2Error):
        m.forward_backward(dtok, dtgt, 9, w["T"], 1.0)        # B > batch_size
    with pytest.raises(G.GPT2Error):
        m.forward_backward(dtok, dtgt, 8, w["T"] + 4, 1.0)    # T > block_size
    with pytest.raises(G.GPT2Error):
        m.forward_backward(dtok, dtgt, 8, w["T"] - 2, 1.0)    # bf16 backward: T % 4
    m.close()


def test_bf16_ragged_batch_and_length():
    """B and T below the handle's sizes, T not a multiple of the 128-row tiles (T % 4 == 0
    for the bf16 backward): loss and every gradient against the oracle."""
    m, params, cfg, w = make("char-bf16", B=8)
    B, T = 3, 100
    tok, tgt = S.batch(w["tok_seed"], 7, B, T, w["V"], w["dist"], w["s"])
    loss = m.forward(torch.tensor(tok).cuda(), torch.tensor(tgt).cuda(), B, T, want_loss=True)
    m.zero_grad()
    m.backward(1.0)
    grads = m.get_grads()
    ref = O.forward(params, cfg, tok, tgt)
    rgrads = O.backward(params, cfg, ref["cache"], 1.0)
    assert abs(loss - ref["loss"]) <= 2e-2, (loss, ref["loss"])
    worst = {k: cosine(grads[k], rgrads[k]) for k in grads if np.abs(rgrads[k]).max() > 0}
    assert min(worst.values()) >= 0.999, worst
    m.close()


def test_forward_backward_graphs_per_shape():
    """Graph replay keeps one graph per (B, T, scale): alternating shapes give the eager
    results."""
    m, params, cfg, w = make("char-bf16", B=8)
    shapes = [(3, 100), (8, 256), (3, 100), (8, 256)]
    batches = []
    for i, (B, T) in enumerate(shapes):
        tok, tgt = S.batch(w["tok_seed"], 20 + i, B, T, w["V"], w["dist"], w["s"])
        batches.append((B, T, torch.tensor(tok).cuda(), torch.tensor(tgt).cuda()))

    def run(graph):
        m.set_params(params)
        m.set_graph_mode(graph)
        m.zero_grad()
        losses = []
        for B, T, dtok, dtgt in batches:
            if graph:
                m.forward_backward(dtok, dtgt, B, T, 0.5)
            else:
                m.forward(dtok, dtgt, B, T)
                m.backward(0.5)
            losses.append(m.get_loss())
        return losses, m.read_region("grads", np.float32)

    l_e, g_e = run(False)
    l_g, g_g = run(True)
    assert l_g == l_e and np.array_equal(g_g, g_e)
    m.close()


def test_checkpoint_resume_is_bit_identical():
    """Checkpoint = the fp32 parameters, both AdamW moments and the step counter. Restored into
    a new handle (writing the parameters refreshes its bf16 copy), the next optimiser step
    gives the same parameters bit for bit as the uninterrupted run."""
    m, params, cfg, w = make("char-bf16", B=8)
    batches = [tokens_for(w, 8, index=30 + i) for i in range(3)]

    def train_step(model, i):
        tok, tgt, dtok, dtgt = batches[i]
        model.zero_grad()
        model.forward_backward(dtok, dtgt, 8, w["T"], 1.0)
        model.adamw_step(1e-3, 0.9, 0.95, 1e-8, 0.1, grad_clip=1.0)

    train_step(m, 0)
    train_step(m, 1)
    ckpt = {r: m.read_region(r, np.float32) for r in ("params", "m", "v")}
    t = m.step
    assert t == 2
    train_step(m, 2)
    want = m.read_region("params", np.float32)

    m2, _, _, _ = make("char-bf16", B=8)
    for r, a in ckpt.items():
        m2.write_region(r, a)
    m2.step = t
    train_step(m2, 2)
    got = m2.read_region("params", np.float32)
    assert not np.array_equal(want, ckpt["params"])   # the step did move the parameters
    assert np.array_equal(got, want)
    m.close()
    m2.close()


def test_bf16_zero_logits_give_ln_vocab():
    """lnf gamma = beta = 0 makes every logit exactly 0: the loss is ln V over the real
    vocabulary (the padded columns are masked)."""
    m, params, cfg, w = make("gpt2-124m-micro", B=1)
    params = dict(params)
    params["lnfw"] = np.zeros_like(params["lnfw"])
    params["lnfb"] = np.zeros_like(params["lnfb"])
    m.set_params(params)
    _, _, dtok, dtgt = tokens_for(w, 1)
    loss = m.forward(dtok, dtgt, want_loss=True)
    assert abs(loss - math.log(50257)) < 1e-5
    m.close()


def test_bf16_causal_invariance():
    m, params, cfg, w = make("char-bf16", B=2)
    tok, tgt, _, _ = tokens_for(w, 2)
    t = 100
    a = m.forward(torch.tensor(tok).cuda(), None)
    za = m.read_region("logits", np.uint16, count=2 * w["T"] * w["Vp"]).reshape(2, w["T"], -1)
    tok2 = tok.copy()
    tok2[:, t + 1:] = (tok2[:, t + 1:] + 7) % w["V"]
    m.forward(torch.tensor(tok2).cuda(), None)
    zb = m.read_region("logits", np.uint16, count=2 * w["T"] * w["Vp"]).reshape(2, w["T"], -1)
    assert np.array_equal(za[:, :t + 1], zb[:, :t + 1])
    assert not np.array_equal(za[:, t + 1:], zb[:, t + 1:])
    m.close()


def test_bf16_argmax_matches_logits():
    m, params, cfg, w = make("char-bf16", B=2)
    tok, _, dtok, _ = tokens_for(w, 2)
    m.forward(dtok, None)
    z = m.read_region("logits", np.uint16, count=2 * w["T"] * w["Vp"]).reshape(-1, w["Vp"])
    zf = (z.astype(np.uint32) << 16).view(np.float32)[:, :w["V"]]
    am = m.read_region("argmax", np.int32, count=2 * w["T"])
    assert np.array_equal(am, zf.argmax(-1))
    m.close()


# ----------------------------------------------------------------- errors
def test_sequence_longer_than_block_size():
    m, params, cfg, w = make("tiny-fp32", B=1)
    x = torch.zeros(1, w["T"] + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(G.GPT2Error) as e:
        m.forward(x, x)
    assert e.value.name == "SEQ_TOO_LONG"
    m.close()


def test_out_of_range_token_is_reported():
    m, params, cfg, w = make("tiny-fp32", B=1)
    x = torch.zeros(1, w["T"], dtype=torch.int32, device="cuda")
    x[0, 5] = w["V"] + 3          # clamped on read, reported at the next sync
    with pytest.raises(G.GPT2Error) as e:
        m.forward(x, x.clamp(0, w["V"] - 1), want_loss=True)
    assert e.value.name == "BAD_TOKEN"
    m.sync()                      # the error word was cleared
    m.close()


def test_backward_needs_forward_with_targets():
    m, params, cfg, w = make("tiny-fp32", B=1)
    with pytest.raises(G.GPT2Error) as e:
        m.backward(1.0)
    assert e.value.name == "STATE"
    m.close()
