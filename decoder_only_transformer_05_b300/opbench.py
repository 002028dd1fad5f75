"""Time single kernels of the training step at the GPT-2 124M shapes (B=12, T=1024,
C=768, H=12, V=50257 padded to 50304) through the op-level C ABI, with CUDA events.

    python -m decoder_only_transformer_05_b300.opbench [--ops gemm,attn,ln,cls,ce,decode] [--iters N]

Each line reports the kernel's average duration and its throughput against the
algorithmic work (2*M*N*K flops for GEMMs, causal attention flops, bytes moved once for
the memory-bound kernels). The device footprint is that of one op (at most ~1.5 GB), so
it is also the small-case command for profiler captures of a single kernel.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import build as _build
from . import gpt2 as G

B, T, C, H, Vp, V = 12, 1024, 768, 12, 50304, 50257
M = B * T


def _linear_shapes():
    # name: (N_out, K_in) of y = x W^T
    return {"qkv": (3 * C, C), "attproj": (C, C), "fc": (4 * C, C), "fcproj": (C, 4 * C),
            "lmhead": (Vp, C)}


def gemm_cases():
    out = []
    for name, (N, K) in _linear_shapes().items():
        epi = "gelu_fwd" if name == "fc" else "store"
        out.append((f"gemm_fwd_{name}", dict(kind="fwd", N=N, K=K, epi=epi)))
        out.append((f"gemm_dgrad_{name}", dict(kind="dgrad", N=N, K=K,
                                               epi="gelu_bwd" if name == "fcproj" else "store")))
        out.append((f"gemm_wgrad_{name}", dict(kind="wgrad", N=N, K=K, epi="accum")))
    return out


def _bf16(*shape):
    return (0.02 * torch.randn(*shape, device="cuda")).to(torch.bfloat16)


def run_gemm(name, kind, N, K, epi, iters):
    if kind == "fwd":
        X, W = _bf16(M, K), _bf16(N, K)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        bias = _bf16(N) if name != "gemm_fwd_lmhead" else None
        pre = torch.empty_like(Y) if epi == "gelu_fwd" else None
        resid = _bf16(M, N) if name in ("gemm_fwd_attproj", "gemm_fwd_fcproj") else None
        args = dict(precision="bf16", M=M, N=N, K=K, A=X, lda=K, a_mn=False, B=W, ldb=K,
                    b_mn=False, epi=epi, out=Y, ldo=N, bias=bias, resid=resid, pre=pre)
        gm, gn, gk = M, N, K
    elif kind == "dgrad":
        dY, W = _bf16(M, N), _bf16(N, K)
        dX = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
        aux = _bf16(M, K) if epi == "gelu_bwd" else None
        args = dict(precision="bf16", M=M, N=K, K=N, A=dY, lda=N, a_mn=False, B=W, ldb=K,
                    b_mn=True, epi=epi, out=dX, ldo=K, aux=aux)
        gm, gn, gk = M, K, N
    else:
        dY, X = _bf16(M, N), _bf16(M, K)
        acc = torch.zeros(N, K, device="cuda")
        ws = torch.empty(16 * N * K if N * K <= 4096 * 1024 else 1, device="cuda")
        args = dict(precision="bf16", M=N, N=K, K=M, A=dY, lda=N, a_mn=True, B=X, ldb=K,
                    b_mn=True, epi="accum", accum=acc, ldo=K, scale=1.0, splits=0,
                    workspace=ws, workspace_bytes=ws.numel() * 4)
        gm, gn, gk = N, K, M
    ms = _time(lambda s: G.op_gemm(**args, stream=s), iters)
    return dict(op=name, ms=ms, tflops=2.0 * gm * gn * gk / (ms * 1e-3) / 1e12,
                shape=[gm, gn, gk])


def run_attention(iters):
    qkv = _bf16(B, T, 3 * C) * 50
    out = torch.empty(B, T, C, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, T, device="cuda")
    dout = _bf16(B, T, C)
    dqkv = torch.empty_like(qkv)
    Dbuf = torch.empty(2, B, H, T, device="cuda")
    flops = 2 * 2 * B * H * (T * (T + 1) / 2) * (C // H)   # causal QK^T and PV
    ms_f = _time(lambda s: G.op_attention_forward("bf16", out, lse, qkv, B, T, C, H, stream=s),
                 iters)
    ms_b = _time(lambda s: G.op_attention_backward("bf16", dqkv, Dbuf, dout, out, qkv, lse, B,
                                                   T, C, H, stream=s), iters)
    return [dict(op="attention_fwd", ms=ms_f, tflops=flops / (ms_f * 1e-3) / 1e12),
            dict(op="attention_bwd", ms=ms_b, tflops=2.5 * flops / (ms_b * 1e-3) / 1e12)]


def run_layernorm(iters):
    x, w, b = _bf16(M, C), _bf16(C), _bf16(C)
    y = torch.empty_like(x)
    mean, rstd = torch.empty(M, device="cuda"), torch.empty(M, device="cuda")
    ms_f = _time(lambda s: G.op_layernorm_forward("bf16", y, mean, rstd, x, w, b, M, C, stream=s),
                 iters)
    dres, dw, db = _bf16(M, C), torch.zeros(C, device="cuda"), torch.zeros(C, device="cuda")
    part = torch.empty(G.op_layernorm_partials_floats(M, C), device="cuda")
    ms_b = _time(lambda s: G.op_layernorm_backward("bf16", dres, 1, dw, db, y, x, w, mean, rstd,
                                                   M, C, 1.0, part, stream=s), iters)
    return [dict(op="layernorm_fwd", ms=ms_f, gbs=(2 * M * C * 2 + 8 * M) / (ms_f * 1e-3) / 1e9),
            dict(op="layernorm_bwd", ms=ms_b,
                 gbs=(4 * M * C * 2 + 8 * M) / (ms_b * 1e-3) / 1e9)]


def run_classifier(iters):
    logits = _bf16(M, Vp) * 100
    tgt = torch.randint(0, V, (M,), dtype=torch.int32, device="cuda")
    losses = torch.empty(M, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ms = _time(lambda s: G.op_classifier("bf16", logits, losses, tgt, M, V, Vp, err, stream=s),
               iters)
    return [dict(op="classifier", ms=ms, gbs=2 * M * Vp * 2 / (ms * 1e-3) / 1e9)]


def run_ce(iters):
    """The lm_head with the cross-entropy statistics in its epilogue plus the combine and the
    streaming dlogits pass, against the plain lm_head GEMM plus the two-pass classifier."""
    x, wte = _bf16(M, C), _bf16(Vp, C)
    tgt = torch.randint(0, V, (M,), dtype=torch.int32, device="cuda")
    logits = torch.empty(M, Vp, dtype=torch.bfloat16, device="cuda")
    losses = torch.empty(M, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.empty(G.op_lmhead_ce_scratch_bytes(M, Vp) // 4 + 4, device="cuda")
    ms_fused = _time(lambda s: G.op_lmhead_cross_entropy(M, C, V, Vp, x, wte, tgt, logits,
                                                         losses, scratch, err, stream=s), iters)

    def unfused(s):
        G.op_gemm("bf16", M, Vp, C, x, C, False, wte, C, False, "store", out=logits, ldo=Vp,
                  stream=s)
        G.op_classifier("bf16", logits, losses, tgt, M, V, Vp, err, stream=s)
    ms_unfused = _time(unfused, iters)
    return [dict(op="lmhead_cross_entropy_fused", ms=ms_fused),
            dict(op="lmhead_then_classifier", ms=ms_unfused)]


def run_decode(iters):
    """Greedy decoding with the key/value cache on the 124M shape: a 512-token prompt per row
    (prefill), then `iters` decode steps of one token per row, for 1 and 12 rows."""
    out = []
    for rows in (1, 12):
        m = G.GPT2(vocab_size=V, padded_vocab_size=Vp, block_size=T, n_layer=12, n_head=H,
                   n_embd=C, batch_size=rows, bias=True, precision="bf16", init=True, seed=5)
        prompt = torch.randint(0, V, (rows, 512), dtype=torch.int32, device="cuda")
        nxt = torch.empty(rows, dtype=torch.int32, device="cuda")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m.prefill(prompt, nxt)
        torch.cuda.synchronize()
        e0.record()
        m.prefill(prompt, nxt)
        e1.record()
        torch.cuda.synchronize()
        ms_pre = e0.elapsed_time(e1)
        steps = min(iters, T - 512 - 1)
        e0.record()
        for _ in range(steps):
            m.decode_step(nxt, nxt)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        out.append(dict(op=f"decode_step_rows{rows}", ms=ms, tokens_per_s=rows / (ms * 1e-3),
                        prefill_ms=ms_pre,
                        # every step reads all bf16 weights once (the lm_head's 77 MB included)
                        weight_gbs=2 * m.num_params / (ms * 1e-3) / 1e9))
        m.close()
    return out


def _time(fn, iters):
    """Average device time of fn(stream) over `iters` back-to-back launches, replayed from a
    CUDA graph so that the host-side cost of each call (argument marshalling, tensor-map
    encoding) does not leave the GPU idle between short kernels."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            fn(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        for _ in range(iters):
            fn(s)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        g.replay()
        e0.record()
        g.replay()
        e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--ops", default="gemm,attn,ln,cls")
    ap.add_argument("--gemm", default="", help="comma list of GEMM case names (default all)")
    ap.add_argument("--iters", type=int, default=10)
    a = ap.parse_args()
    _build.build()
    G.load_library()
    torch.manual_seed(0)
    ops = a.ops.split(",")
    rows = []
    if "gemm" in ops:
        sel = set(a.gemm.split(",")) if a.gemm else None
        for name, kw in gemm_cases():
            if sel is None or name in sel:
                rows.append(run_gemm(name, iters=a.iters, **kw))
                torch.cuda.empty_cache()
    if "attn" in ops:
        rows += run_attention(a.iters)
    if "ln" in ops:
        rows += run_layernorm(a.iters)
    if "cls" in ops:
        rows += run_classifier(a.iters)
    if "ce" in ops:
        rows += run_ce(a.iters)
    if "decode" in ops:
        rows += run_decode(max(a.iters, 64))
    for r in rows:
        print(json.dumps(r))


if __name__ == "__main__":
    main()
