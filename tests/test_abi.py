"""CPU checks of the C-ABI library: it loads, exports every entry point the headers
declare, validates configurations, and its host-side initialiser and parameter counts
agree with the seeded generator and the oracle. No kernel runs here."""
import os
import re
import subprocess

import numpy as np
import pytest
import torch

from decoder_only_transformer_05_b300 import build as B
from decoder_only_transformer_05_b300 import gpt2 as G
from decoder_only_transformer_05_b300 import synthetic as S
from oracle import gpt2_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return G.load_library()


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(gpt2_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = declared_symbols()
    assert len(declared) >= 25
    out = subprocess.run(["nm", "-D", "--defined-only", G.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (gpt2_\w+)", out))
    assert declared <= exported, declared - exported
    assert declared == set(G.SIGNATURES), declared ^ set(G.SIGNATURES)
    for name in declared:
        assert getattr(lib, name) is not None


def test_library_is_built_for_sm_103a():
    # the link step embeds device code for sm_103a only (cuobjdump is not used: the
    # architecture list is read from the build flags the library was produced with)
    assert "arch=compute_103a,code=sm_103a" in " ".join(B.ARCH)


@pytest.mark.parametrize("name", list(S.WORKLOADS))
def test_parameter_counts_match_oracle(lib, name):
    w = S.WORKLOADS[name]
    n_model, n_buf = G.host_num_params(vocab_size=w["V"], padded_vocab_size=w["Vp"],
                                       block_size=w["T"], n_layer=w["L"], n_head=w["H"],
                                       n_embd=w["C"], batch_size=w["B"], bias=w["bias"],
                                       precision=w["precision"])
    cfg = O.Config(w["V"], w["Vp"], w["T"], w["L"], w["H"], w["C"], w["bias"])
    assert n_model == O.num_parameters(cfg)
    assert n_buf >= O.num_parameters(cfg, padded=True)


@pytest.mark.parametrize("name", ["tiny-fp32", "char-bf16"])
def test_host_init_matches_seeded_generator(lib, name):
    """gpt2_create's initialiser (C++) and synthetic.init_params (numpy) implement the same
    counter-mode SplitMix64 + Box-Muller definition."""
    w = S.WORKLOADS[name]
    kw = dict(vocab_size=w["V"], padded_vocab_size=w["Vp"], block_size=w["T"],
              n_layer=w["L"], n_head=w["H"], n_embd=w["C"], batch_size=w["B"],
              bias=w["bias"], precision=w["precision"], seed=w["w_seed"])
    flat = G.host_init(**kw)
    ref = S.init_params(w["w_seed"], w["V"], w["Vp"], w["T"], w["L"], w["C"], w["bias"])
    # offsets: each tensor starts on a 64-float boundary, in table order
    off = 0
    for _, name_, shape, _ in S.param_table(w["V"], w["Vp"], w["T"], w["L"], w["C"], w["bias"]):
        n = int(np.prod(shape))
        np.testing.assert_allclose(flat[off:off + n].reshape(shape), ref[name_], rtol=2e-7,
                                   atol=1e-12, err_msg=name_)
        off += (n + 63) // 64 * 64
    assert off == flat.size


@pytest.mark.parametrize("bad", [dict(n_embd=100, n_head=3), dict(vocab_size=0),
                                 dict(padded_vocab_size=10), dict(n_head=4, n_embd=128),
                                 dict(batch_size=0)])
def test_invalid_configs_are_rejected(lib, bad):
    kw = dict(vocab_size=65, padded_vocab_size=128, block_size=64, n_layer=2, n_head=2,
              n_embd=128, batch_size=2, precision="bf16")
    kw.update(bad)
    with pytest.raises(G.GPT2Error) as e:
        G.host_num_params(**kw)
    assert e.value.name == "INVALID_CONFIG"
    with pytest.raises(G.GPT2Error) as e:
        G.GPT2(**kw)
    assert e.value.name == "INVALID_CONFIG"


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_create_without_gpu_fails_cleanly(lib):
    with pytest.raises(G.GPT2Error) as e:
        G.GPT2(vocab_size=65, block_size=64, n_layer=1, n_head=2, n_embd=128, batch_size=1,
               precision="fp32")
    assert e.value.name in ("CUDA", "OOM")
