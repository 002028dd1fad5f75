"""Greedy inference with the key/value cache (gpt2_prefill, gpt2_decode_step) against the
oracle: at every generated position the GPU's logits (computed from the cache) match the
oracle's forward over the whole sequence so far, the token the GPU chose is the argmax of
its own logits bit for bit (lowest index on ties, the same bf16/fp32 values), and that
token is a valid greedy choice for the oracle (its logit within the logits' tolerance of
the maximum). The generation loop is that of 「从零实现一个最小GPT」 三.8 (argmax instead of
sampling).
"""
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


def make(name, B):
    w = S.WORKLOADS[name]
    m = G.GPT2(vocab_size=w["V"], padded_vocab_size=w["Vp"], block_size=w["T"],
               n_layer=w["L"], n_head=w["H"], n_embd=w["C"], batch_size=B, bias=w["bias"],
               precision=w["precision"], init=False)
    params = S.init_params(w["w_seed"], w["V"], w["Vp"], w["T"], w["L"], w["C"], w["bias"])
    m.set_params(params)
    cfg = O.Config(w["V"], w["Vp"], w["T"], w["L"], w["H"], w["C"], w["bias"])
    return m, params, cfg, w


def logits_rows(m, w, rows):
    if w["precision"] == "fp32":
        return m.read_region("logits", np.float32, count=rows * w["Vp"]).reshape(rows, -1)
    z = m.read_region("logits", np.uint16, count=rows * w["Vp"]).reshape(rows, -1)
    return (z.astype(np.uint32) << 16).view(np.float32)


def cosine(a, r):
    a, r = np.asarray(a, np.float64).reshape(-1), np.asarray(r, np.float64).reshape(-1)
    return float(a @ r / (np.linalg.norm(a) * np.linalg.norm(r) + 1e-300))


# B = 20 takes the tensor-core GEMMs and the separate LayerNorm / cache-store kernels (the
# weight-streaming kernel with its fusions handles at most 16 rows)
@pytest.mark.parametrize("name,B,T0,n_new", [("tiny-fp32", 2, 16, 8), ("char-bf16", 3, 50, 20),
                                             ("char-bf16", 20, 30, 5),
                                             ("gpt2-124m-micro", 1, 100, 4)])
def test_greedy_decode_matches_oracle(name, B, T0, n_new):
    m, params, cfg, w = make(name, B)
    V = w["V"]
    fp32 = w["precision"] == "fp32"
    prompt, _ = S.batch(w["tok_seed"], 9, B, T0, V, w["dist"], w["s"])
    seq = prompt.copy()
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    m.prefill(torch.tensor(prompt).cuda(), nxt)
    gpu_logits = []
    z = logits_rows(m, w, B * T0).reshape(B, T0, -1)[:, -1, :V]
    gpu_logits.append(z)
    for i in range(n_new):
        tok = nxt.cpu().numpy()
        assert np.array_equal(tok, gpu_logits[-1].argmax(-1))   # bit-exact argmax
        seq = np.concatenate([seq, tok[:, None]], axis=1)
        if i + 1 < n_new:
            m.decode_step(nxt.clone(), nxt)
            assert m.decode_length == T0 + i + 1
            gpu_logits.append(logits_rows(m, w, B)[:, :V])
    # the oracle over the growing sequence: its last-position logits at each step
    for i, z in enumerate(gpu_logits):
        ref = O.forward(params, cfg, seq[:, :T0 + i])["logits"][:, -1, :]
        if fp32:
            assert np.abs(z - ref).max() <= 1e-4 * max(np.abs(ref).max(), 1.0), i
        else:
            for b in range(B):
                assert cosine(z[b], ref[b]) >= 0.9999, (i, b)
            assert np.abs(z - ref).max() <= 5e-2, i
        chosen = seq[:, T0 + i]
        gap = ref.max(-1) - ref[np.arange(B), chosen]
        assert (gap <= (1e-4 if fp32 else 5e-2)).all(), (i, gap)
    m.close()


def test_decode_cache_matches_a_full_forward():
    """The decode path's logits at each new position against the ordinary forward over the
    whole sequence on the same GPU (same precision, different kernels and blocking: each is
    within the bf16 logits bound of the oracle, cosine >= 0.9999, and so is the pair)."""
    m, params, cfg, w = make("char-bf16", 2)
    B, T0, n_new, V = 2, 64, 16, w["V"]
    prompt, _ = S.batch(w["tok_seed"], 11, B, T0, V, w["dist"], w["s"])
    out = m.generate(torch.tensor(prompt).cuda(), n_new).cpu().numpy()
    seq = np.concatenate([prompt, out], axis=1)
    dec = []
    m.prefill(torch.tensor(prompt).cuda(), torch.empty(B, dtype=torch.int32, device="cuda"))
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    for i in range(n_new - 1):
        m.decode_step(torch.tensor(out[:, i].copy()).cuda(), nxt)
        dec.append(logits_rows(m, w, B)[:, :V])
    T = T0 + n_new - 1
    m.forward(torch.tensor(seq[:, :T].copy()).cuda(), None, B, T)
    full = logits_rows(m, w, B * T).reshape(B, T, -1)[:, :, :V]
    assert m.decode_length == 0          # the ordinary forward discarded the cache
    for i, z in enumerate(dec):
        for b in range(B):
            assert cosine(z[b], full[b, T0 + i]) >= 0.9999, (i, b)
    m.close()


def test_decode_errors():
    m, params, cfg, w = make("char-bf16", 2)
    nxt = torch.empty(2, dtype=torch.int32, device="cuda")
    tok = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(G.GPT2Error) as e:
        m.decode_step(tok, nxt)                      # no prefill
    assert e.value.name == "STATE"
    full = torch.zeros(2, w["T"], dtype=torch.int32, device="cuda")
    m.prefill(full, nxt)                             # the whole block
    with pytest.raises(G.GPT2Error) as e:
        m.decode_step(tok, nxt)
    assert e.value.name == "SEQ_TOO_LONG"
    m.prefill(full[:, :10].contiguous(), nxt)
    with pytest.raises(G.GPT2Error) as e:
        m.decode_step(tok[:1].contiguous(), nxt)     # B differs from the prefill's
    assert e.value.name == "ARG"
    m.close()


@pytest.mark.parametrize("name,B", [("char-bf16", 2), ("gpt2-124m-micro", 12)])
def test_replayed_decode_steps_match_eager_ones(name, B):
    """After its first step for a batch, gpt2_decode_step replays a recorded graph whose
    kernels read the position from device memory; the tokens and logits it produces are
    bit-identical to those of the same steps run eagerly (graph mode off)."""
    w = S.WORKLOADS[name]
    T0, n_new = 40, 12
    prompt, _ = S.batch(w["tok_seed"], 13, B, T0, w["V"], w["dist"], w["s"])
    runs = []
    for graph in (True, False):
        m, params, cfg, w = make(name, B)
        m.set_graph_mode(graph)
        nxt = torch.empty(B, dtype=torch.int32, device="cuda")
        m.prefill(torch.tensor(prompt).cuda(), nxt)
        toks, logits = [], []
        for i in range(n_new):
            m.decode_step(nxt.clone(), nxt)
            toks.append(nxt.cpu().numpy().copy())
            logits.append(m.read_region("logits", np.uint16 if w["precision"] != "fp32" else np.float32,
                                        count=B * w["Vp"]).copy())
        runs.append((toks, logits))
        m.close()
    for a, b in zip(runs[0][0], runs[1][0]):
        assert np.array_equal(a, b)
    for a, b in zip(runs[0][1], runs[1][1]):
        assert np.array_equal(a, b)
