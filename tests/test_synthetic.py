"""The seeded input generators: published SplitMix64 outputs, ranges, the next-token
shift, Zipf frequencies and the entropy floor of each workload."""
import math

import numpy as np

from decoder_only_transformer_05_b300 import synthetic as S


def test_splitmix64_published_first_output():
    # SplitMix64 seeded with 0: the first output is 0xE220A8397B1DCDAF
    assert int(S.draw(0, np.array([0], dtype=np.uint64))[0]) == 0xE220A8397B1DCDAF


def test_uniform_and_normal_moments():
    u = S.uniform(S.stream_key(3, 0), 200000)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.005
    n = S.normal(S.stream_key(3, 1), 200000)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1.0) < 0.01


def test_targets_are_tokens_shifted_by_one():
    tok, tgt = S.batch(0, 0, 4, 64, 65)
    assert tok.dtype == np.int32 and tok.shape == (4, 64)
    assert np.array_equal(tok[:, 1:], tgt[:, :-1])
    assert tok.min() >= 0 and tok.max() < 65


def test_batches_differ_and_repeat():
    a = S.batch(2, 0, 2, 16, 50257, "zipf", 1.0)
    b = S.batch(2, 1, 2, 16, 50257, "zipf", 1.0)
    c = S.batch(2, 0, 2, 16, 50257, "zipf", 1.0)
    assert not np.array_equal(a[0], b[0])
    assert np.array_equal(a[0], c[0])


def test_zipf_frequencies_and_entropy_floor():
    V, s = 50257, 1.0
    ids = S.token_stream(2, 0, 64, 1024, V, "zipf", s).reshape(-1)
    p = np.arange(1, V + 1, dtype=np.float64) ** -s
    p /= p.sum()
    # id 0 carries about 8.8% of the tokens
    assert abs(p[0] - 0.0880) < 5e-4
    assert abs((ids == 0).mean() - p[0]) < 4 * math.sqrt(p[0] / ids.size)
    H = -(p * np.log(p)).sum()
    assert abs(H - 7.5659) < 1e-3
    p65 = np.arange(1, 66, dtype=np.float64) ** -1.1
    p65 /= p65.sum()
    assert abs(-(p65 * np.log(p65)).sum() - 3.1948) < 1e-3


def test_init_params_layout():
    p = S.init_params(1000, 65, 128, 64, 4, 128, bias=False)
    assert set(p) == {"wte", "wpe", "ln1w", "ln1b", "qkvw", "attprojw", "ln2w", "ln2b",
                      "fcw", "fcprojw", "lnfw", "lnfb"}
    assert p["wte"].shape == (128, 128) and np.all(p["wte"][65:] == 0)
    assert abs(p["wte"][:65].std() - 0.02) < 0.002
    assert abs(p["fcprojw"].std() - 0.02 / math.sqrt(8)) < 0.0005
    assert np.all(p["ln1w"] == 1) and np.all(p["lnfb"] == 0)
