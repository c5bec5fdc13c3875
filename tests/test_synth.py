"""The seeded generators produce the block structure the recipe states."""
import numpy as np

from quant_quantized_matvec_gb300 import synth


def test_deterministic_and_seed_sensitive():
    a = synth.kquant_matrix(synth.Q4_K, 3, 512, "t/a")
    b = synth.kquant_matrix(synth.Q4_K, 3, 512, "t/a")
    c = synth.kquant_matrix(synth.Q4_K, 3, 512, "t/b")
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    assert a.shape == (3, 2 * 144)


def test_q45_headers():
    for fmt, bb in ((synth.Q4_K, 144), (synth.Q5_K, 176)):
        W = synth.kquant_matrix(fmt, 64, 1024, f"t/{fmt}")
        blocks = W.reshape(-1, bb)
        hdr = blocks[:, 0:4].copy().view(np.float16).astype(np.float64)
        assert hdr.min() >= np.float16(1e-3) and hdr.max() <= np.float16(1e-2)
        # the payload bytes are uniform: all byte values occur
        assert len(np.unique(blocks[:, 4:])) == 256


def test_q6_fields():
    W = synth.kquant_matrix(synth.Q6_K, 64, 1024, "t/q6")
    blocks = W.reshape(-1, 210)
    sc = blocks[:, 192:208].copy().view(np.int8)
    assert sc.min() == -32 and sc.max() == 31
    d = blocks[:, 208:210].copy().view(np.float16).astype(np.float64)
    assert d.min() >= np.float16(1e-3) and d.max() <= np.float16(1e-2)
    assert len(np.unique(blocks[:, :192])) == 256


def test_activations():
    x = synth.activations(8, 6656, "t/x")
    assert x.dtype == np.float32 and x.shape == (8, 6656)
    assert abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1) < 0.05
