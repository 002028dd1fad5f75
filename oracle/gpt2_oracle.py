"""CPU oracle for one GPT-2 training step: forward, hand-written backward,
global-norm clip and AdamW, in float64 numpy.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or run this
module: only the tests, the smoke check and the CPU-baseline leg of the benchmark
use it. It shares no code with the CUDA library (it never imports the package).

What it follows (cited by page title and section):
  * 「从零实现一个最小GPT：代码讲解 + 知识点全解」 (a minimal GPT in PyTorch), sections
    二.3-二.7 and 三.3-三.7: token plus position embedding, pre-LN blocks
    x += attn(LN1 x); x += mlp(LN2 x), per-head causal softmax(q k^T / sqrt(head_size)) v
    with the heads concatenated in head order, a 4x MLP, final LayerNorm, lm_head, and a
    mean cross-entropy over all B*T positions whose target is the next token (三.2).
  * 「两小时手搓GPT-2：Karpathy用124M参数打脸“黑盒神话”」, section "Attention、MLP与那个
    容易被忽略的GELU近似": GPT-2's GELU is an approximation, not the exact form.
  * 「手写训练脚本：不用框架，从零实现GPT训练流程」, sections 二-三: each layer's backward
    written out by hand and chained; parameters in one flat buffer.
  * 「从零实现一个最小GPT」 section 三.9: AdamW (adaptive step plus decoupled weight
    decay) over all parameters.
  * 「4.1 GPT-2 (124M) 复现」 section 2.3: gradient accumulation and the 6e-4 -> 6e-5
    learning-rate range with 2000 warmup steps.

Readings where the pages are silent or disagree:
  * fused QKV: one [3C, C] weight whose rows are the Q, K, V thirds, each third
    holding the heads in order; equal to the per-head Linears stacked.
  * the lm_head is tied to the token embedding; logits cover the first V (unpadded)
    columns only.
  * LayerNorm: biased variance, eps 1e-5, gamma and beta always present; the bias flag
    covers the Linear layers only.
  * tanh-GELU: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) (Hendrycks and
    Gimpel 2016).
  * AdamW as PyTorch documents it (bias-corrected moments, eps added after the
    square root, step count from 1); clip coefficient min(1, c / (||g|| + 1e-6)).

Parity pins: see tests/test_oracle_pins.py (finite differences, torch CPU autograd in
float64, loss = ln V for zero logits, attention rows, causal invariance, GELU bounds
against the exact erf form, parameter counts, torch.optim.AdamW).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

LN_EPS = 1e-5
GELU_K = math.sqrt(2.0 / math.pi)
GELU_C = 0.044715


@dataclass
class Config:
    vocab_size: int
    padded_vocab_size: int
    block_size: int
    n_layer: int
    n_head: int
    n_embd: int
    bias: bool = True


def parameter_shapes(cfg: Config):
    """Ordered (name, shape) list of every parameter, padded wte rows included."""
    V, Vp, T, L, C = (cfg.vocab_size, cfg.padded_vocab_size, cfg.block_size,
                      cfg.n_layer, cfg.n_embd)
    shapes = [("wte", (Vp, C)), ("wpe", (T, C)),
              ("ln1w", (L, C)), ("ln1b", (L, C)),
              ("qkvw", (L, 3 * C, C)), ("qkvb", (L, 3 * C)),
              ("attprojw", (L, C, C)), ("attprojb", (L, C)),
              ("ln2w", (L, C)), ("ln2b", (L, C)),
              ("fcw", (L, 4 * C, C)), ("fcb", (L, 4 * C)),
              ("fcprojw", (L, C, 4 * C)), ("fcprojb", (L, C)),
              ("lnfw", (C,)), ("lnfb", (C,))]
    if not cfg.bias:
        shapes = [s for s in shapes if s[0] not in ("qkvb", "attprojb", "fcb", "fcprojb")]
    return shapes


def num_parameters(cfg: Config, padded: bool = False) -> int:
    n = sum(int(np.prod(s)) for _, s in parameter_shapes(cfg))
    if not padded:
        n -= (cfg.padded_vocab_size - cfg.vocab_size) * cfg.n_embd
    return n


# ----------------------------------------------------------------------------------
# elementary layers (forward and backward), float64

def encoder_forward(wte, wpe, tokens):
    """x[b, t] = wte[tokens[b, t]] + wpe[t] (「从零实现一个最小GPT」 三.7, forward step 1)."""
    T = tokens.shape[1]
    return wte[tokens] + wpe[:T][None, :, :]


def encoder_backward(dx, tokens, Vp):
    """Scatter-add of dx into the token rows; sum over the batch for positions."""
    B, T, C = dx.shape
    dwte = np.zeros((Vp, C))
    np.add.at(dwte, tokens.reshape(-1), dx.reshape(-1, C))
    dwpe = dx.sum(axis=0)
    return dwte, dwpe


def layernorm_forward(x, w, b):
    """(x - mean) / sqrt(var + eps) * w + b over the last axis, biased variance."""
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + LN_EPS)
    xhat = (x - mean) * rstd
    return xhat * w + b, mean[..., 0], rstd[..., 0]


def layernorm_backward(dy, x, w, mean, rstd):
    """Chain rule through the normalisation (「手写训练脚本」 二: LayerNorm's backward
    derived by hand). Returns dx, dw, db (dw, db summed over rows)."""
    xhat = (x - mean[..., None]) * rstd[..., None]
    dxhat = dy * w
    C = x.shape[-1]
    dx = rstd[..., None] * (dxhat - dxhat.sum(-1, keepdims=True) / C
                            - xhat * (dxhat * xhat).sum(-1, keepdims=True) / C)
    dw = (dy * xhat).reshape(-1, C).sum(0)
    db = dy.reshape(-1, C).sum(0)
    return dx, dw, db


def gelu(x):
    return 0.5 * x * (1.0 + np.tanh(GELU_K * (x + GELU_C * x ** 3)))


def gelu_grad(x):
    t = np.tanh(GELU_K * (x + GELU_C * x ** 3))
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * GELU_K * (1.0 + 3.0 * GELU_C * x * x)


def _split_heads(qkv, H):
    """qkv [B, T, 3C] -> q, k, v each [B, H, T, hs]; head h is columns h*hs..(h+1)*hs
    of its third (「从零实现一个最小GPT」 三.4: heads concatenated in order)."""
    B, T, C3 = qkv.shape
    C = C3 // 3
    hs = C // H
    q, k, v = qkv[..., :C], qkv[..., C:2 * C], qkv[..., 2 * C:]
    f = lambda a: a.reshape(B, T, H, hs).transpose(0, 2, 1, 3)
    return f(q), f(k), f(v)


def attention_weights(q, k):
    """Causal softmax(q k^T / sqrt(hs)) for [.., T, hs] inputs (「从零实现一个最小GPT」
    三.3: scores, future positions set to -inf, softmax over keys)."""
    T, hs = q.shape[-2], q.shape[-1]
    s = (q @ np.swapaxes(k, -1, -2)) * (1.0 / math.sqrt(hs))
    future = np.triu(np.ones((T, T), dtype=bool), k=1)
    s = np.where(future, -np.inf, s)
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


def attention_forward(qkv, H):
    """out [B, T, C] (heads concatenated) and the weights P [B, H, T, T]."""
    B, T, C3 = qkv.shape
    q, k, v = _split_heads(qkv, H)
    P = attention_weights(q, k)
    o = P @ v
    return o.transpose(0, 2, 1, 3).reshape(B, T, C3 // 3), P


def attention_backward(dout, qkv, P, H):
    """d qkv from d out: dV = P^T dO, dP = dO V^T, dS = P (dP - rowsum(P dP)),
    dQ = dS K / sqrt(hs), dK = dS^T Q / sqrt(hs)."""
    B, T, C3 = qkv.shape
    C = C3 // 3
    hs = C // H
    q, k, v = _split_heads(qkv, H)
    do = dout.reshape(B, T, H, hs).transpose(0, 2, 1, 3)
    dv = np.swapaxes(P, -1, -2) @ do
    dP = do @ np.swapaxes(v, -1, -2)
    dS = P * (dP - (P * dP).sum(-1, keepdims=True))
    scale = 1.0 / math.sqrt(hs)
    dq = (dS @ k) * scale
    dk = (np.swapaxes(dS, -1, -2) @ q) * scale
    g = lambda a: a.transpose(0, 2, 1, 3).reshape(B, T, C)
    return np.concatenate([g(dq), g(dk), g(dv)], axis=-1)


def cross_entropy_forward(logits, targets):
    """Per-position loss logsumexp(z) - z[y] and softmax probabilities."""
    zmax = logits.max(-1, keepdims=True)
    e = np.exp(logits - zmax)
    ssum = e.sum(-1, keepdims=True)
    lse = (np.log(ssum) + zmax)[..., 0]
    probs = e / ssum
    zy = np.take_along_axis(logits, targets[..., None], axis=-1)[..., 0]
    return lse - zy, probs


# ----------------------------------------------------------------------------------
# the model

def _lin(x, w, b):
    y = x @ w.T
    return y if b is None else y + b


def forward(params: dict, cfg: Config, tokens: np.ndarray, targets=None):
    """One forward pass. Returns dict(loss, losses [B,T], logits [B,T,V], cache)."""
    p = {k: np.asarray(v, dtype=np.float64) for k, v in params.items()}
    B, T = tokens.shape
    if T > cfg.block_size:
        raise ValueError("sequence longer than block_size")
    V, L, H = cfg.vocab_size, cfg.n_layer, cfg.n_head
    bias = (lambda n, l: p[n][l]) if cfg.bias else (lambda n, l: None)
    tokens = np.asarray(tokens, dtype=np.int64)
    if tokens.min() < 0 or tokens.max() >= V:
        raise ValueError("token id out of range")
    x = encoder_forward(p["wte"], p["wpe"], tokens)
    cache = dict(tokens=tokens, x0=x, layers=[])
    for l in range(L):
        c = dict(x_in=x)
        c["h1"], c["m1"], c["r1"] = layernorm_forward(x, p["ln1w"][l], p["ln1b"][l])
        c["qkv"] = _lin(c["h1"], p["qkvw"][l], bias("qkvb", l))
        c["att"], c["P"] = attention_forward(c["qkv"], H)
        x = x + _lin(c["att"], p["attprojw"][l], bias("attprojb", l))
        c["x_mid"] = x
        c["h2"], c["m2"], c["r2"] = layernorm_forward(x, p["ln2w"][l], p["ln2b"][l])
        c["u"] = _lin(c["h2"], p["fcw"][l], bias("fcb", l))
        c["a"] = gelu(c["u"])
        x = x + _lin(c["a"], p["fcprojw"][l], bias("fcprojb", l))
        cache["layers"].append(c)
    cache["x_L"] = x
    xf, mf, rf = layernorm_forward(x, p["lnfw"], p["lnfb"])
    cache.update(xf=xf, mf=mf, rf=rf)
    logits = xf @ p["wte"][:V].T
    out = dict(logits=logits, cache=cache, loss=None, losses=None)
    if targets is not None:
        targets = np.asarray(targets, dtype=np.int64)
        losses, probs = cross_entropy_forward(logits, targets)
        out.update(losses=losses, loss=float(losses.mean()))
        cache.update(targets=targets, probs=probs)
    return out


def backward(params: dict, cfg: Config, cache: dict, loss_scale: float = 1.0) -> dict:
    """Gradients of loss_scale * mean loss with respect to every parameter."""
    p = {k: np.asarray(v, dtype=np.float64) for k, v in params.items()}
    V, Vp, L, H = cfg.vocab_size, cfg.padded_vocab_size, cfg.n_layer, cfg.n_head
    tokens, targets, probs = cache["tokens"], cache["targets"], cache["probs"]
    B, T = tokens.shape
    g = {name: np.zeros(shape) for name, shape in parameter_shapes(cfg)}

    dlogits = probs.copy()
    np.put_along_axis(dlogits, targets[..., None],
                      np.take_along_axis(dlogits, targets[..., None], -1) - 1.0, -1)
    dlogits *= loss_scale / (B * T)
    C = cfg.n_embd
    g["wte"][:V] += dlogits.reshape(-1, V).T @ cache["xf"].reshape(-1, C)
    dxf = dlogits @ p["wte"][:V]
    dx, g["lnfw"], g["lnfb"] = layernorm_backward(dxf, cache["x_L"], p["lnfw"],
                                                  cache["mf"], cache["rf"])
    for l in reversed(range(L)):
        c = cache["layers"][l]
        # x_out = x_mid + a Wp^T + bp
        g["fcprojw"][l] = dx.reshape(-1, C).T @ c["a"].reshape(-1, 4 * C)
        if cfg.bias:
            g["fcprojb"][l] = dx.reshape(-1, C).sum(0)
        da = dx @ p["fcprojw"][l]
        du = da * gelu_grad(c["u"])
        g["fcw"][l] = du.reshape(-1, 4 * C).T @ c["h2"].reshape(-1, C)
        if cfg.bias:
            g["fcb"][l] = du.reshape(-1, 4 * C).sum(0)
        dh2 = du @ p["fcw"][l]
        dx2, g["ln2w"][l], g["ln2b"][l] = layernorm_backward(dh2, c["x_mid"], p["ln2w"][l],
                                                             c["m2"], c["r2"])
        dx = dx + dx2
        # x_mid = x_in + att Wo^T + bo
        g["attprojw"][l] = dx.reshape(-1, C).T @ c["att"].reshape(-1, C)
        if cfg.bias:
            g["attprojb"][l] = dx.reshape(-1, C).sum(0)
        datt = dx @ p["attprojw"][l]
        dqkv = attention_backward(datt, c["qkv"], c["P"], H)
        g["qkvw"][l] = dqkv.reshape(-1, 3 * C).T @ c["h1"].reshape(-1, C)
        if cfg.bias:
            g["qkvb"][l] = dqkv.reshape(-1, 3 * C).sum(0)
        dh1 = dqkv @ p["qkvw"][l]
        dx1, g["ln1w"][l], g["ln1b"][l] = layernorm_backward(dh1, c["x_in"], p["ln1w"][l],
                                                             c["m1"], c["r1"])
        dx = dx + dx1
    dwte, dwpe = encoder_backward(dx, tokens, Vp)
    g["wte"] += dwte
    g["wpe"][:T] += dwpe
    return g


# ----------------------------------------------------------------------------------
# optimiser

def global_norm(grads: dict) -> float:
    return math.sqrt(sum(float((np.asarray(a, np.float64) ** 2).sum()) for a in grads.values()))


def clip_coefficient(grads: dict, max_norm: float):
    """(||g||_2, min(1, max_norm / (||g|| + 1e-6))); max_norm <= 0 disables clipping."""
    n = global_norm(grads)
    if max_norm <= 0:
        return n, 1.0
    return n, min(1.0, max_norm / (n + 1e-6))


def adamw_update(p, g, m, v, t, lr, beta1, beta2, eps, weight_decay, grad_scale=1.0):
    """One AdamW step on arrays (t counts from 1). Returns new (p, m, v)."""
    p = np.asarray(p, np.float64)
    g = np.asarray(g, np.float64) * grad_scale
    m = beta1 * np.asarray(m, np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, np.float64) + (1.0 - beta2) * g * g
    p = p * (1.0 - lr * weight_decay)
    mhat = m / (1.0 - beta1 ** t)
    vhat = v / (1.0 - beta2 ** t)
    p = p - lr * mhat / (np.sqrt(vhat) + eps)
    return p, m, v


def lr_warmup_cosine(it, max_lr=6e-4, min_lr=6e-5, warmup=2000, max_iters=600000):
    """Linear warmup (it+1)/warmup, then cosine from max_lr down to min_lr at
    max_iters, constant after (values from 「4.1 GPT-2 (124M) 复现」 2.3)."""
    if it < warmup:
        return max_lr * (it + 1) / warmup
    if it >= max_iters:
        return min_lr
    ratio = (it - warmup) / (max_iters - warmup)
    return min_lr + 0.5 * (1.0 + math.cos(math.pi * ratio)) * (max_lr - min_lr)


def lr_cosine(it, max_lr=1e-3, min_lr=1e-4, total=100):
    """Cosine decay without warmup, min_lr = max_lr / 10."""
    it = min(it, total)
    return min_lr + 0.5 * (1.0 + math.cos(math.pi * it / total)) * (max_lr - min_lr)


def training_step(params, m, v, t, cfg, micro_batches, lr, beta1, beta2, eps,
                  weight_decay, grad_clip):
    """One optimiser step: accumulate gradients of loss/accum over the micro-batches,
    clip, AdamW. Returns (new params, m, v, mean loss, grad norm, grads)."""
    accum = len(micro_batches)
    grads = {name: np.zeros(shape) for name, shape in parameter_shapes(cfg)}
    losses = []
    for tok, tgt in micro_batches:
        out = forward(params, cfg, tok, tgt)
        losses.append(out["loss"])
        gi = backward(params, cfg, out["cache"], 1.0 / accum)
        for k in grads:
            grads[k] += gi[k]
    norm, coef = clip_coefficient(grads, grad_clip)
    newp, newm, newv = {}, {}, {}
    for k in params:
        newp[k], newm[k], newv[k] = adamw_update(params[k], grads[k], m[k], v[k], t, lr,
                                                 beta1, beta2, eps, weight_decay, coef)
    return newp, newm, newv, float(np.mean(losses)), norm, grads
