"""Per-kernel parity on the GPU, through the C ABI (include/gpt2_ops.h), against the CPU
oracle in float64 on the same (bf16-rounded, for the bf16 path) inputs."""
import math

import numpy as np
import pytest
import torch

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
    torch.cuda.init()
    yield


def dev(a, dtype):
    return torch.tensor(np.asarray(a), dtype=torch.float32).to(dtype).cuda().contiguous()


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).normal(0.0, scale, size=shape)


def rel_inf(a, r):
    return float(np.abs(a - r).max() / max(np.abs(r).max(), 1e-30))


def cosine(a, r):
    a, r = a.reshape(-1), r.reshape(-1)
    return float(a @ r / (np.linalg.norm(a) * np.linalg.norm(r) + 1e-300))


# ------------------------------------------------------------------------ GEMM
# (M, N, K): several tiles, ragged M, both BN widths (N % 256 == 0 -> 256, else 128)
SHAPES = [(256, 384, 192), (200, 256, 128), (384, 768, 256), (130, 128, 64),
          (200, 256, 136)]   # ragged K: the last k-block reads zeros past K


def gemm_ref(A, B_, a_mn, b_mn):
    Am = A.T if a_mn else A       # -> [M, K]
    Bm = B_.T if b_mn else B_     # -> [N, K]
    return Am @ Bm.T


@pytest.mark.parametrize("prec", ["bf16", "fp32"])
@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, True), (True, False)])
@pytest.mark.parametrize("shape", SHAPES)
def test_gemm_store(prec, a_mn, b_mn, shape):
    M, N, K = shape
    dt = torch.bfloat16 if prec == "bf16" else torch.float32
    # an MN-major A is stored [K, lda] with lda padded to a multiple of 8 elements
    lda = (M + 7) // 8 * 8 if a_mn else K
    A = rnd((K, lda) if a_mn else (M, K), 1)
    Bm = rnd((K, N) if b_mn else (N, K), 2)
    bias = rnd((N,), 3)
    resid = rnd((M, N), 4)
    dA, dB, db, dr = dev(A, dt), dev(Bm, dt), dev(bias, dt), dev(resid, dt)
    out = torch.empty(M, N, dtype=dt, device="cuda")
    G.op_gemm(prec, M, N, K, dA, lda, a_mn, dB, N if b_mn else K, b_mn, "store",
              out=out, ldo=N, bias=db, resid=dr)
    torch.cuda.synchronize()
    Ah = host(dA)[:, :M] if a_mn else host(dA)
    ref = gemm_ref(Ah, host(dB), a_mn, b_mn) + host(db)[None, :] + host(dr)
    got = host(out)
    if prec == "bf16":
        assert rel_inf(got, ref) < 8e-3
        assert np.all(np.abs(got - ref) <= 2 ** -8 * np.abs(ref) + 2e-3 * np.abs(ref).max())
    else:
        assert rel_inf(got, ref) < 1e-5


@pytest.mark.parametrize("prec", ["bf16", "fp32"])
def test_gemm_gelu_fwd_and_bwd(prec):
    M, N, K = 256, 512, 192
    dt = torch.bfloat16 if prec == "bf16" else torch.float32
    X, W, b = dev(rnd((M, K), 5), dt), dev(rnd((N, K), 6, 0.1), dt), dev(rnd((N,), 7), dt)
    out = torch.empty(M, N, dtype=dt, device="cuda")
    pre = torch.empty(M, N, dtype=dt, device="cuda")
    G.op_gemm(prec, M, N, K, X, K, False, W, K, False, "gelu_fwd", out=out, ldo=N, bias=b,
              pre=pre)
    torch.cuda.synchronize()
    u = host(X) @ host(W).T + host(b)[None, :]
    tol = 8e-3 if prec == "bf16" else 1e-5
    # `pre` keeps gelu'(u), what the backward multiplies by
    assert rel_inf(host(pre), O.gelu_grad(u)) < tol
    assert rel_inf(host(out), O.gelu(u)) < tol
    # dgrad with the GELU derivative: out = (dY W) * pre
    dY = dev(rnd((M, K), 8), dt)
    d = torch.empty(M, N, dtype=dt, device="cuda")
    # dgrad layout: d[M, N] = dY[M, K] W2[K, N] with W2 MN-major
    W2 = dev(rnd((K, N), 9, 0.1), dt)
    G.op_gemm(prec, M, N, K, dY, K, False, W2, N, True, "gelu_bwd", out=d, ldo=N, aux=pre)
    torch.cuda.synchronize()
    ref = (host(dY) @ host(W2)) * host(pre)
    assert rel_inf(host(d), ref) < (1.5e-2 if prec == "bf16" else 1e-5)


@pytest.mark.parametrize("prec", ["bf16", "fp32"])
def test_gemm_gelu_epilogues_for_recomputation(prec):
    """The recomputation pair: the forward keeps u = X W^T + b (and writes gelu(u)); the
    backward's dgrad multiplies by gelu'(u) recomputed from u and writes gelu(u) again (for
    the weight gradient). Ragged M and 3 column tiles."""
    M, N, K = 300, 384, 128
    dt = torch.bfloat16 if prec == "bf16" else torch.float32
    X, W, b = dev(rnd((M, K), 15), dt), dev(rnd((N, K), 16, 0.1), dt), dev(rnd((N,), 17), dt)
    out = torch.empty(M, N, dtype=dt, device="cuda")
    u = torch.empty(M, N, dtype=dt, device="cuda")
    G.op_gemm(prec, M, N, K, X, K, False, W, K, False, "gelu_fwd_u", out=out, ldo=N, bias=b,
              pre=u)
    torch.cuda.synchronize()
    ref_u = host(X) @ host(W).T + host(b)[None, :]
    tol = 8e-3 if prec == "bf16" else 1e-5
    assert rel_inf(host(u), ref_u) < tol
    assert rel_inf(host(out), O.gelu(ref_u)) < tol
    dY = dev(rnd((M, K), 18), dt)
    W2 = dev(rnd((K, N), 19, 0.1), dt)
    d = torch.empty(M, N, dtype=dt, device="cuda")
    g = torch.empty(M, N, dtype=dt, device="cuda")
    G.op_gemm(prec, M, N, K, dY, K, False, W2, N, True, "gelu_bwd_u", out=d, ldo=N, aux=u, pre=g)
    torch.cuda.synchronize()
    uu = host(u)   # the kept (rounded) pre-activation is what the backward sees
    assert rel_inf(host(d), (host(dY) @ host(W2)) * O.gelu_grad(uu)) < (1.5e-2 if prec == "bf16" else 1e-5)
    assert rel_inf(host(g), O.gelu(uu)) < tol


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("shape", [(384, 256, 1024), (768, 768, 4096), (384, 256, 300)])
def test_gemm_wgrad_accumulate_bf16(splits, shape):
    """dW[N, K] += scale * dY^T X with both operands MN-major, split-K partials reduced in
    a fixed order."""
    Mtok, Nout, Kin = shape[2], shape[0], shape[1]
    dY = dev(rnd((Mtok, Nout), 10), torch.bfloat16)
    X = dev(rnd((Mtok, Kin), 11), torch.bfloat16)
    acc0 = rnd((Nout, Kin), 12)
    acc = torch.tensor(acc0, dtype=torch.float32, device="cuda")
    ws = torch.empty(16 * Nout * Kin, dtype=torch.float32, device="cuda")
    G.op_gemm("bf16", Nout, Kin, Mtok, dY, Nout, True, X, Kin, True, "accum", accum=acc, ldo=Kin,
              scale=0.25, splits=splits, workspace=ws, workspace_bytes=ws.numel() * 4)
    torch.cuda.synchronize()
    ref = acc0.astype(np.float32).astype(np.float64) + 0.25 * (host(dY).T @ host(X))
    got = acc.cpu().numpy().astype(np.float64)
    assert rel_inf(got, ref) < 2e-5


def test_gemm_rejects_unaligned_sizes():
    x = torch.zeros(64 * 130, dtype=torch.bfloat16, device="cuda")
    # N not a multiple of 64
    with pytest.raises(G.GPT2Error) as e:
        G.op_gemm("bf16", 64, 48, 64, x, 64, False, x, 64, False, "store", out=x, ldo=64)
    assert e.value.name == "ARG"
    # leading dimension of an MN-major operand not a multiple of 8 elements
    with pytest.raises(G.GPT2Error) as e:
        G.op_gemm("bf16", 130, 64, 64, x, 130, True, x, 64, False, "store", out=x, ldo=64)
    assert e.value.name == "ARG"


@pytest.mark.parametrize("epi", ["store", "gelu_fwd"])
def test_gemm_partial_last_wide_tile(epi):
    """N = 16.5 x 256 (as the padded vocabulary, 50304 = 196.5 x 256) keeps 256-wide tiles:
    the last tile's B rows past N read as zero and its columns past N are not stored.
    Ragged M as well."""
    M, N, K = 200, 4224, 128
    X, W, b = dev(rnd((M, K), 13), torch.bfloat16), dev(rnd((N, K), 14, 0.1), torch.bfloat16), \
        dev(rnd((N,), 15), torch.bfloat16)
    out = torch.full((M, N + 64), 7.0, dtype=torch.bfloat16, device="cuda")
    pre = torch.full((M, N + 64), 7.0, dtype=torch.bfloat16, device="cuda")
    G.op_gemm("bf16", M, N, K, X, K, False, W, K, False, epi, out=out, ldo=N + 64, bias=b,
              pre=pre if epi == "gelu_fwd" else None)
    torch.cuda.synchronize()
    u = host(X) @ host(W).T + host(b)[None, :]
    ref = O.gelu(u) if epi == "gelu_fwd" else u
    assert rel_inf(host(out)[:, :N], ref) < 8e-3
    assert torch.all(out[:, N:] == 7.0)          # the padding columns are untouched
    if epi == "gelu_fwd":
        assert rel_inf(host(pre)[:, :N], O.gelu_grad(u)) < 8e-3
        assert torch.all(pre[:, N:] == 7.0)


def test_gemm_large_forward_shape():
    """The 124M model's QKV projection at full size (M = 12 x 1024 tokens), row-sampled."""
    M, N, K = 12288, 2304, 768
    X = torch.randn(M, K, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16).cuda()
    W = (0.02 * torch.randn(N, K, generator=torch.Generator().manual_seed(1))).to(
        torch.bfloat16).cuda()
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    G.op_gemm("bf16", M, N, K, X, K, False, W, K, False, "store", out=out, ldo=N)
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(M, 64, replace=False)
    ref = host(X)[rows] @ host(W).T
    assert rel_inf(host(out)[rows], ref) < 8e-3


# ------------------------------------------------------------------- attention
@pytest.mark.parametrize("B,T,H,hs", [(2, 256, 2, 64), (1, 1024, 12, 64), (2, 100, 3, 64),
                                      (3, 388, 2, 64)])
def test_attention_bf16(B, T, H, hs):
    C = H * hs
    qkv = dev(rnd((B, T, 3 * C), 20), torch.bfloat16)
    out = torch.empty(B, T, C, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    G.op_attention_forward("bf16", out, lse, qkv, B, T, C, H)
    dout = dev(rnd((B, T, C), 21), torch.bfloat16)
    dqkv = torch.zeros(B, T, 3 * C, dtype=torch.bfloat16, device="cuda")
    Dbuf = torch.empty(2, B, H, T, dtype=torch.float32, device="cuda")
    G.op_attention_backward("bf16", dqkv, Dbuf, dout, out, qkv, lse, B, T, C, H)
    torch.cuda.synchronize()
    q = host(qkv)
    ref_out, P = O.attention_forward(q, H)
    assert rel_inf(host(out), ref_out) < 2e-2
    assert cosine(host(out), ref_out) > 0.9999
    qq, kk, _ = O._split_heads(q, H)
    s = (qq @ np.swapaxes(kk, -1, -2)) / math.sqrt(hs)
    s = np.where(np.triu(np.ones((T, T), bool), 1), -np.inf, s)
    ref_lse = np.log(np.exp(s - s.max(-1, keepdims=True)).sum(-1)) + s.max(-1)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=0, atol=2e-3)
    ref_d = O.attention_backward(host(dout), q, P, H)
    got = host(dqkv)
    for part in range(3):
        sl = slice(part * C, (part + 1) * C)
        assert cosine(got[..., sl], ref_d[..., sl]) > 0.999, part
        assert rel_inf(got[..., sl], ref_d[..., sl]) < 3e-2, part


def test_attention_bf16_backward_rejects_t_not_multiple_of_4():
    B, T, H, C = 1, 66, 1, 64
    qkv = torch.zeros(B, T, 3 * C, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(B, T, C, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, H, T, dtype=torch.float32, device="cuda")
    dqkv = torch.zeros_like(qkv)
    Dbuf = torch.zeros(2, B, H, T, dtype=torch.float32, device="cuda")
    with pytest.raises(G.GPT2Error) as e:
        G.op_attention_backward("bf16", dqkv, Dbuf, out, out, qkv, lse, B, T, C, H)
    assert e.value.name == "ARG"


def test_attention_fp32():
    B, T, H, C = 2, 64, 4, 128
    qkv = dev(rnd((B, T, 3 * C), 22), torch.float32)
    out = torch.empty(B, T, C, device="cuda")
    lse = torch.empty(B, H, T, device="cuda")
    G.op_attention_forward("fp32", out, lse, qkv, B, T, C, H)
    dout = dev(rnd((B, T, C), 23), torch.float32)
    dqkv = torch.zeros(B, T, 3 * C, device="cuda")
    Dbuf = torch.empty(2, B, H, T, device="cuda")
    G.op_attention_backward("fp32", dqkv, Dbuf, dout, out, qkv, lse, B, T, C, H)
    torch.cuda.synchronize()
    ref_out, P = O.attention_forward(host(qkv), H)
    assert rel_inf(host(out), ref_out) < 1e-5
    ref_d = O.attention_backward(host(dout), host(qkv), P, H)
    assert rel_inf(host(dqkv), ref_d) < 1e-4


# ------------------------------------------------------------------- layernorm
@pytest.mark.parametrize("prec,M,C", [("bf16", 300, 768), ("bf16", 64, 384), ("fp32", 96, 128),
                                      ("bf16", 33, 1024)])
def test_layernorm(prec, M, C):
    dt = torch.bfloat16 if prec == "bf16" else torch.float32
    x = dev(rnd((M, C), 30, 2.0) + 0.5, dt)
    w = dev(1.0 + rnd((C,), 31, 0.2), dt)
    b = dev(rnd((C,), 32, 0.2), dt)
    y = torch.empty(M, C, dtype=dt, device="cuda")
    mean = torch.empty(M, device="cuda")
    rstd = torch.empty(M, device="cuda")
    G.op_layernorm_forward(prec, y, mean, rstd, x, w, b, M, C)
    dy = dev(rnd((M, C), 33), dt)
    dres0 = rnd((M, C), 34)
    dres = dev(dres0, dt)
    dw = torch.zeros(C, device="cuda")
    db = torch.zeros(C, device="cuda")
    part = torch.empty(G.op_layernorm_partials_floats(M, C), device="cuda")
    G.op_layernorm_backward(prec, dres, 1, dw, db, dy, x, w, mean, rstd, M, C, 0.5, part)
    torch.cuda.synchronize()
    ry, rm, rr = O.layernorm_forward(host(x), host(w), host(b))
    tol = 1e-2 if prec == "bf16" else 1e-5
    assert rel_inf(host(y), ry) < tol
    np.testing.assert_allclose(mean.cpu().numpy(), rm, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(rstd.cpu().numpy(), rr, rtol=1e-4)
    rdx, rdw, rdb = O.layernorm_backward(host(dy), host(x), host(w), rm, rr)
    base = dres0.astype(np.float32) if prec == "fp32" else host(dev(dres0, dt))
    assert rel_inf(host(dres), base + rdx) < tol
    assert rel_inf(dw.cpu().numpy(), 0.5 * rdw) < 1e-4
    assert rel_inf(db.cpu().numpy(), 0.5 * rdb) < 1e-4


# ------------------------------------------------------------------ classifier
@pytest.mark.parametrize("prec,M,V,Vp", [("bf16", 64, 65, 128), ("fp32", 48, 65, 128),
                                         ("bf16", 16, 50257, 50304)])
def test_classifier(prec, M, V, Vp):
    dt = torch.bfloat16 if prec == "bf16" else torch.float32
    z = rnd((M, Vp), 40, 3.0)
    z[:, V:] = 50.0      # pad columns must be ignored even when large
    logits = dev(z, dt)
    zin = host(logits)[:, :V]
    tgt = np.random.default_rng(41).integers(0, V, size=M).astype(np.int32)
    losses = torch.empty(M, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.op_classifier(prec, logits, losses, torch.tensor(tgt).cuda(), M, V, Vp, err)
    torch.cuda.synchronize()
    rl, probs = O.cross_entropy_forward(zin, tgt.astype(np.int64))
    np.testing.assert_allclose(losses.cpu().numpy(), rl, rtol=0, atol=1e-4)
    d = probs.copy()
    d[np.arange(M), tgt] -= 1.0
    d /= M
    got = host(logits)
    tol = 1e-2 if prec == "bf16" else 1e-5
    assert rel_inf(got[:, :V], d) < tol
    assert np.all(got[:, V:] == 0.0)
    assert int(err.item()) == 0


@pytest.mark.parametrize("M,C,V,Vp", [(300, 128, 1000, 1088), (1024, 768, 50257, 50304)])
def test_lmhead_cross_entropy_fused(M, C, V, Vp):
    """The lm_head GEMM with the softmax statistics in its epilogue, then one pass for the
    losses and dlogits, against the oracle's cross-entropy of the same bf16 logits; the pad
    rows of wte are set large so the pad logits are large, and must still be ignored."""
    x = dev(rnd((M, C), 50, 1.0), torch.bfloat16)
    w = rnd((Vp, C), 51, 0.1)
    w[V:] = 0.5                       # pad logits ~ 0.5 * sum(x): large
    wte = dev(w, torch.bfloat16)
    tgt = np.random.default_rng(52).integers(0, V, size=M).astype(np.int32)
    logits = torch.empty(M, Vp, dtype=torch.bfloat16, device="cuda")
    losses = torch.empty(M, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.empty(G.op_lmhead_ce_scratch_bytes(M, Vp) // 4 + 4, device="cuda")
    G.op_lmhead_cross_entropy(M, C, V, Vp, x, wte, torch.tensor(tgt).cuda(), logits, losses,
                              scratch, err)
    # the same logits through the plain GEMM, rounded to bf16 as the fused one rounds them
    z = torch.empty(M, Vp, dtype=torch.bfloat16, device="cuda")
    G.op_gemm("bf16", M, Vp, C, x, C, False, wte, C, False, "store", out=z, ldo=Vp)
    torch.cuda.synchronize()
    zb = host(z)
    assert np.abs(zb[:, V:]).max() > 10.0          # the pad logits are large
    rl, probs = O.cross_entropy_forward(zb[:, :V], tgt.astype(np.int64))
    np.testing.assert_allclose(losses.cpu().numpy(), rl, rtol=0, atol=1e-4)
    d = probs.copy()
    d[np.arange(M), tgt] -= 1.0
    d /= M
    got = host(logits)
    assert rel_inf(got[:, :V], d) < 1e-2
    assert np.all(got[:, V:] == 0.0)
    assert int(err.item()) == 0
