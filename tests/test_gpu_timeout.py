"""Failure detection on the GPU without a fault: a bounded device-side wait that runs out.

Every mbarrier wait of the tensor-core kernels gives up after a time limit, records
GPT2_ERR_TIMEOUT in the handle's device error word, lets the block's own copies and MMAs
finish, frees its tensor memory and returns. The test hook gpt2_debug_gemm_waits shortens
the GEMM's limit to a few milliseconds and withholds one arrival (the signal that a block
pair's first accumulator is ready), so the epilogue's wait runs out. The host must read
GPT2_ERR_TIMEOUT at the next sync, and the same handle must then train on normally: the
next forward's loss equals the one before the fault, bit for bit.
"""
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
    gpt2.debug_gemm_waits(0, False)


def test_gemm_wait_that_runs_out_is_reported_and_the_handle_recovers():
    w = S.WORKLOADS["char-bf16"]
    B = 2
    m = G.GPT2(vocab_size=w["V"], padded_vocab_size=w["Vp"], block_size=w["T"],
               n_layer=w["L"], n_head=w["H"], n_embd=w["C"], batch_size=B, bias=w["bias"],
               precision="bf16", init=True, seed=w["w_seed"])
    tok, tgt = S.batch(w["tok_seed"], 0, B, w["T"], w["V"], w["dist"], w["s"])
    dtok, dtgt = torch.tensor(tok).cuda(), torch.tensor(tgt).cuda()
    before = m.forward(dtok, dtgt, want_loss=True)
    try:
        G.debug_gemm_waits(5_000_000, True)      # 5 ms limit, one arrival withheld
        m.forward(dtok, dtgt)                    # queued; nothing waits on the host
    finally:
        G.debug_gemm_waits(0, False)
    with pytest.raises(G.GPT2Error) as e:
        m.sync()
    assert e.value.name == "TIMEOUT"
    m.sync()                                     # the error word was cleared
    after = m.forward(dtok, dtgt, want_loss=True)
    assert after == before
    m.zero_grad()
    m.backward(1.0)
    g = m.read_region("grads", np.float32)
    assert np.isfinite(g).all() and np.abs(g).max() > 0
    m.close()
