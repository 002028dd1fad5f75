"""Pins for the CPU oracle: each test ties it to something other than itself
(finite differences, torch's own CPU implementation in float64, closed forms, the
pages' worked examples and invariants)."""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import gpt2_oracle as O
from decoder_only_transformer_05_b300 import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny_cfg(bias=True, V=11, Vp=16, T=5, L=2, H=2, C=8):
    return O.Config(vocab_size=V, padded_vocab_size=Vp, block_size=T, n_layer=L,
                    n_head=H, n_embd=C, bias=bias)


def random_params(cfg, seed=0, scale=0.3):
    """Non-trivial parameters (LayerNorm gains and biases random too), pad rows 0."""
    rng = np.random.default_rng(seed)
    p = {}
    for name, shape in O.parameter_shapes(cfg):
        a = rng.normal(0.0, scale, size=shape)
        if name in ("ln1w", "ln2w", "lnfw"):
            a = 1.0 + a
        p[name] = a
    p["wte"][cfg.vocab_size:] = 0.0
    return p


def tiny_batch(cfg, B=2, seed=1):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, cfg.vocab_size, size=(B, cfg.block_size + 1))
    return ids[:, :-1], ids[:, 1:]


# --------------------------------------------------------------------------- FD

@pytest.mark.parametrize("bias", [True, False])
def test_backward_matches_central_differences(bias):
    cfg = tiny_cfg(bias=bias)
    p = random_params(cfg)
    tok, tgt = tiny_batch(cfg)
    out = O.forward(p, cfg, tok, tgt)
    g = O.backward(p, cfg, out["cache"], 1.0)
    h = 1e-6
    for name, _ in O.parameter_shapes(cfg):
        flat = p[name].reshape(-1)
        fd = np.zeros_like(flat)
        for i in range(flat.size):
            if name == "wte" and i >= cfg.vocab_size * cfg.n_embd:
                continue     # padded rows never reach the loss
            old = flat[i]
            flat[i] = old + h
            lp = O.forward(p, cfg, tok, tgt)["loss"]
            flat[i] = old - h
            lm = O.forward(p, cfg, tok, tgt)["loss"]
            flat[i] = old
            fd[i] = (lp - lm) / (2 * h)
        an = g[name].reshape(-1)
        err = np.abs(an - fd).max() / max(np.abs(fd).max(), 1e-12)
        assert err <= 1e-6, (name, err)


def test_loss_scale_is_linear():
    cfg = tiny_cfg()
    p = random_params(cfg)
    tok, tgt = tiny_batch(cfg)
    out = O.forward(p, cfg, tok, tgt)
    g1 = O.backward(p, cfg, out["cache"], 1.0)
    g4 = O.backward(p, cfg, out["cache"], 0.25)
    for k in g1:
        np.testing.assert_allclose(g4[k], 0.25 * g1[k], rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------ torch in float64

def torch_reference(p, cfg, tok, tgt):
    """The same model written with torch's own CPU routines (layer_norm,
    scaled_dot_product_attention with is_causal, gelu approximate='tanh', cross_entropy)
    and differentiated by autograd, float64."""
    tp = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    V, C, H, L = cfg.vocab_size, cfg.n_embd, cfg.n_head, cfg.n_layer
    B, T = tok.shape
    idx = torch.tensor(tok)
    x = F.embedding(idx, tp["wte"]) + tp["wpe"][:T]
    b = (lambda n, l: tp[n][l]) if cfg.bias else (lambda n, l: None)
    for l in range(L):
        h = F.layer_norm(x, (C,), tp["ln1w"][l], tp["ln1b"][l], eps=1e-5)
        qkv = F.linear(h, tp["qkvw"][l], b("qkvb", l))
        q, k, v = qkv.split(C, dim=-1)
        sh = lambda a: a.view(B, T, H, C // H).transpose(1, 2)
        y = F.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True)
        y = y.transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(y, tp["attprojw"][l], b("attprojb", l))
        h = F.layer_norm(x, (C,), tp["ln2w"][l], tp["ln2b"][l], eps=1e-5)
        u = F.gelu(F.linear(h, tp["fcw"][l], b("fcb", l)), approximate="tanh")
        x = x + F.linear(u, tp["fcprojw"][l], b("fcprojb", l))
    x = F.layer_norm(x, (C,), tp["lnfw"], tp["lnfb"], eps=1e-5)
    logits = F.linear(x, tp["wte"][:V])
    loss = F.cross_entropy(logits.reshape(-1, V), torch.tensor(tgt).reshape(-1))
    loss.backward()
    return loss.item(), logits.detach().numpy(), {k: t.grad.numpy() for k, t in tp.items()}


@pytest.mark.parametrize("bias,shape", [(True, dict()), (False, dict()),
                                        (True, dict(V=65, Vp=128, T=16, L=3, H=4, C=32))])
def test_matches_torch_autograd_fp64(bias, shape):
    cfg = tiny_cfg(bias=bias, **shape)
    p = random_params(cfg, seed=3, scale=0.2)
    tok, tgt = tiny_batch(cfg, B=3, seed=4)
    out = O.forward(p, cfg, tok, tgt)
    g = O.backward(p, cfg, out["cache"], 1.0)
    loss, logits, tg = torch_reference(p, cfg, tok, tgt)
    assert abs(out["loss"] - loss) <= 1e-12 * abs(loss)
    np.testing.assert_allclose(out["logits"], logits, rtol=0, atol=1e-12)
    for k in g:
        ref = tg[k]
        err = np.abs(g[k] - ref).max() / max(np.abs(ref).max(), 1e-300)
        assert err <= 1e-10, (k, err)


# ----------------------------------------------------------------- closed forms

@pytest.mark.parametrize("V,Vp,expected", [(65, 128, 4.174387269895637),
                                           (50257, 50304, 10.82490511970208)])
def test_zero_logits_give_ln_vocab(V, Vp, expected):
    """lnf gamma = beta = 0 makes every logit 0, so the loss is ln V over the real
    vocabulary (not ln Vp: the padded columns are masked), and d lnf_beta has the
    closed form sum_bt (mean_v wte[v] - wte[y_bt]) / (B T)."""
    cfg = O.Config(vocab_size=V, padded_vocab_size=Vp, block_size=4, n_layer=1,
                   n_head=2, n_embd=8, bias=True)
    p = random_params(cfg, seed=5, scale=0.1)
    p["lnfw"][:] = 0.0
    p["lnfb"][:] = 0.0
    rng = np.random.default_rng(6)
    ids = rng.integers(0, V, size=(2, 5))
    tok, tgt = ids[:, :-1], ids[:, 1:]
    out = O.forward(p, cfg, tok, tgt)
    assert abs(out["loss"] - math.log(V)) < 1e-12
    assert abs(out["loss"] - expected) < 1e-12
    g = O.backward(p, cfg, out["cache"], 1.0)
    wte = p["wte"][:V]
    closed = (wte.mean(0)[None, :] - wte[tgt.reshape(-1)]).sum(0) / tgt.size
    np.testing.assert_allclose(g["lnfb"], closed, rtol=0, atol=1e-14)
    assert np.all(g["wte"][V:] == 0.0)


def test_parameter_count_closed_form():
    """12 L C^2 + 13 L C + 2 C + (V + T) C with Linear biases; 124,439,808 for the
    GPT-2 124M shape of 「4.1 GPT-2 (124M) 复现」 2.3 (n_layer 12, n_head 12, n_embd 768,
    block_size 1024, vocab 50257)."""
    def closed(V, T, L, C, bias):
        return 12 * L * C * C + (13 if bias else 4) * L * C + 2 * C + (V + T) * C
    cases = [(50257, 50304, 1024, 12, 12, 768, True, 124_439_808),
             (65, 128, 64, 4, 4, 128, False, 805_248),
             (65, 128, 256, 6, 6, 384, True, 10_770_816),
             (50257, 50304, 1024, 24, 16, 1024, True, 354_823_168)]
    for V, Vp, T, L, H, C, bias, n in cases:
        cfg = O.Config(V, Vp, T, L, H, C, bias)
        assert O.num_parameters(cfg) == closed(V, T, L, C, bias) == n
        assert O.num_parameters(cfg, padded=True) == n + (Vp - V) * C


# ------------------------------------------------------------------- attention

def _read_golden(name):
    blocks, cur = {}, None
    for line in open(os.path.join(GOLDEN, name), encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line[0].isalpha():
            cur = line.split()[0]
            blocks[cur] = [line.split()[1:]] if len(line.split()) > 1 else []
            continue
        blocks[cur].append([float(v) for v in line.split()])
    return blocks


def test_attention_worked_example():
    g = _read_golden("attention_worked_example.txt")
    scores = np.array(g["scores"])
    weights = np.array(g["weights"])
    tril = np.array(g["tril"])
    T = scores.shape[0]
    # q = scores * sqrt(T) and k = I give q k^T / sqrt(hs) = scores (hs = T here)
    P = O.attention_weights(scores * math.sqrt(T), np.eye(T))
    assert np.all(P[np.triu_indices(T, 1)] == 0.0)
    assert P[0, 0] == 1.0
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(P, weights, rtol=0, atol=0.025)
    assert np.array_equal(np.tril(np.ones((4, 4))), tril)


def test_attention_rows_and_first_position():
    rng = np.random.default_rng(7)
    B, T, H, C = 2, 9, 3, 12
    qkv = rng.normal(size=(B, T, 3 * C))
    out, P = O.attention_forward(qkv, H)
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.triu(np.ones((T, T)), 1)[None, None] * P == 0.0)
    # position 0 sees only itself: its output is exactly its value vector
    assert np.array_equal(out[:, 0, :], qkv[:, 0, 2 * C:])


def test_causal_invariance():
    """Changing tokens after position t leaves logits and losses at positions <= t
    bit-identical (the causal mask of 「从零实现一个最小GPT」 三.3)."""
    cfg = tiny_cfg(V=13, Vp=16, T=8, L=2, H=2, C=8)
    p = random_params(cfg, seed=8, scale=0.3)
    rng = np.random.default_rng(9)
    ids = rng.integers(0, 13, size=(2, 9))
    tok, tgt = ids[:, :-1].copy(), ids[:, 1:].copy()
    a = O.forward(p, cfg, tok, tgt)
    t = 3
    tok2, tgt2 = tok.copy(), tgt.copy()
    tok2[:, t + 1:] = (tok2[:, t + 1:] + 5) % 13
    tgt2[:, t + 1:] = (tgt2[:, t + 1:] + 7) % 13
    b = O.forward(p, cfg, tok2, tgt2)
    assert np.array_equal(a["logits"][:, :t + 1], b["logits"][:, :t + 1])
    assert np.array_equal(a["losses"][:, :t + 1], b["losses"][:, :t + 1])
    assert not np.array_equal(a["logits"][:, t + 1:], b["logits"][:, t + 1:])


def test_shape_chain():
    """Intermediate shapes follow the table in 「从零实现一个最小GPT」 四."""
    cfg = tiny_cfg(V=11, Vp=16, T=6, L=1, H=2, C=8)
    p = random_params(cfg)
    tok, tgt = tiny_batch(cfg, B=3)
    out = O.forward(p, cfg, tok, tgt)
    B, T, C, hs, V = 3, 6, 8, 4, 11
    sym = dict(B=B, T=T, C=C, hs=hs, V=V)
    shapes = {}
    for line in open(os.path.join(GOLDEN, "shape_chain.txt"), encoding="utf-8"):
        if line.strip() and not line.startswith("#"):
            name, *dims = line.split()
            shapes[name] = tuple(sym[d] for d in dims)
    c = out["cache"]["layers"][0]
    q, k, v = O._split_heads(c["qkv"], 2)
    assert tok.shape == shapes["idx"]
    assert out["cache"]["x0"].shape == shapes["x"] == shapes["tok_emb"]
    assert p["wpe"][:T].shape == shapes["pos_emb"]
    assert q[:, 0].shape == shapes["q"] and k[:, 0].shape == shapes["k"]
    assert c["P"][:, 0].shape == shapes["wei"]
    assert c["att"].shape == shapes["cat"]
    assert c["att"][..., :hs].shape == shapes["out"]
    assert c["u"][..., :C].shape == shapes["ffn"]
    assert out["logits"].shape == shapes["logits"]


def test_sequence_longer_than_block_size_is_rejected():
    cfg = tiny_cfg()
    p = random_params(cfg)
    tok = np.zeros((1, cfg.block_size + 1), dtype=np.int64)
    with pytest.raises(ValueError):
        O.forward(p, cfg, tok)


# ------------------------------------------------------------------------ GELU

def test_gelu_is_the_tanh_approximation():
    """Pinned against torch's gelu(approximate='tanh') and against the exact erf form:
    the approximation differs from x Phi(x) by at most 4.8e-4 (and by more than 1e-4
    near x = 1, so it is not the exact form), and it is odd up to x:
    gelu(x) - gelu(-x) = x."""
    from scipy.special import erf
    x = np.linspace(-8, 8, 4001)
    g = O.gelu(x)
    tg = F.gelu(torch.tensor(x), approximate="tanh").numpy()
    np.testing.assert_allclose(g, tg, rtol=0, atol=1e-15)
    exact = 0.5 * x * (1 + erf(x / math.sqrt(2)))
    d = np.abs(g - exact)
    assert d.max() < 4.8e-4
    assert abs(O.gelu(1.0) - 0.5 * (1 + erf(1 / math.sqrt(2)))) > 1e-4
    np.testing.assert_allclose(O.gelu(x) - O.gelu(-x), x, rtol=0, atol=1e-14)
    assert O.gelu(0.0) == 0.0
    h = 1e-6
    fd = (O.gelu(x + h) - O.gelu(x - h)) / (2 * h)
    np.testing.assert_allclose(O.gelu_grad(x), fd, rtol=0, atol=1e-8)


# --------------------------------------------------------------------- AdamW

def test_adamw_and_clip_match_torch():
    rng = np.random.default_rng(10)
    shapes = [(7, 5), (11,), (3, 4, 2)]
    ps = [rng.normal(size=s) for s in shapes]
    tps = [torch.tensor(p.copy(), requires_grad=True) for p in ps]
    opt = torch.optim.AdamW(tps, lr=1e-2, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    m = [np.zeros(s) for s in shapes]
    v = [np.zeros(s) for s in shapes]
    for t in range(1, 5):
        gs = [rng.normal(size=s) * (3.0 if t == 2 else 0.2) for s in shapes]
        norm, coef = O.clip_coefficient({str(i): g for i, g in enumerate(gs)}, 1.0)
        for tp, g in zip(tps, gs):
            tp.grad = torch.tensor(g.copy())
        tnorm = torch.nn.utils.clip_grad_norm_(tps, 1.0)
        assert abs(norm - float(tnorm)) < 1e-12 * norm
        opt.step()
        for i in range(len(ps)):
            ps[i], m[i], v[i] = O.adamw_update(ps[i], gs[i], m[i], v[i], t, 1e-2, 0.9, 0.95,
                                               1e-8, 0.1, coef)
            np.testing.assert_allclose(ps[i], tps[i].detach().numpy(), rtol=0, atol=1e-14)


def test_clip_disabled_and_small_norm():
    g = {"a": np.array([0.3, 0.4])}
    assert O.clip_coefficient(g, 0.0) == (0.5, 1.0)
    n, c = O.clip_coefficient(g, 1.0)
    assert n == 0.5 and c == 1.0
    n, c = O.clip_coefficient({"a": np.array([3.0, 4.0])}, 1.0)
    assert abs(c - 1.0 / (5.0 + 1e-6)) < 1e-15


def test_lr_schedules():
    """Warmup to 6e-4 over 2000 steps, cosine to 6e-5 at 600000 (「4.1 GPT-2 (124M) 复现」 2.3)."""
    f = O.lr_warmup_cosine
    assert abs(f(0) - 6e-4 / 2000) < 1e-18
    assert abs(f(1999) - 6e-4) < 1e-18
    assert abs(f(2000) - 6e-4) < 1e-18
    assert abs(f(301000) - 0.5 * (6e-4 + 6e-5)) < 1e-15
    assert abs(f(600000) - 6e-5) < 1e-18 and f(10 ** 7) == 6e-5
    assert all(f(i) >= f(i + 1) for i in range(2000, 600000, 997))
    g = O.lr_cosine
    assert abs(g(0) - 1e-3) < 1e-18 and abs(g(100) - 1e-4) < 1e-18
    assert abs(g(50) - 5.5e-4) < 1e-15


def test_training_step_accumulation_equals_big_batch():
    """Accumulating loss/accum over two micro-batches gives the gradient of the mean
    over their union (the gradient-accumulation reading)."""
    cfg = tiny_cfg()
    p = random_params(cfg, seed=11, scale=0.2)
    tok, tgt = tiny_batch(cfg, B=4, seed=12)
    z = {k: np.zeros_like(a) for k, a in p.items()}
    _, _, _, loss2, _, g2 = O.training_step(p, z, z, 1, cfg, [(tok[:2], tgt[:2]),
                                                             (tok[2:], tgt[2:])],
                                            1e-3, 0.9, 0.95, 1e-8, 0.1, 0.0)
    out = O.forward(p, cfg, tok, tgt)
    g1 = O.backward(p, cfg, out["cache"], 1.0)
    assert abs(loss2 - out["loss"]) < 1e-12
    for k in g1:
        np.testing.assert_allclose(g2[k], g1[k], rtol=0, atol=1e-13)
