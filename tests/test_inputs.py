"""The seeded input generators: deterministic, with the stated shapes and structure."""
import numpy as np

from row_wise_softmax_warp_gb300 import inputs


def test_deterministic_and_seed_dependent():
    a = inputs.softmax_pair(0)
    b = inputs.softmax_pair(0)
    c = inputs.softmax_pair(1)
    assert np.array_equal(a["x"], b["x"]) and np.array_equal(a["dy"], b["dy"])
    assert not np.array_equal(a["x"], c["x"])
    assert a["x"].shape == (256, 128) and a["x"].dtype == np.float32
    assert abs(a["x"].std() - 2.0) < 0.05 and abs(a["dy"].std() - 1.0) < 0.03


def test_layernorm_rows():
    d = inputs.layernorm(0, rows=512, cols=768)
    x = d["x"].astype(np.float64)
    s = x.std(axis=1)
    c = x.mean(axis=1)
    assert d["x"].dtype == np.float32 and d["gamma"].shape == (768,)
    assert 0.05 < s.min() and s.max() < 11 and -5.5 < c.min() and c.max() < 5.5
    assert abs(d["gamma"].mean() - 1) < 0.02 and abs(d["beta"].std() - 0.1) < 0.02


def test_cross_entropy_outliers_and_targets():
    d = inputs.cross_entropy(0, rows=64, cols=5000)
    x = d["logits"]
    n = int(round(1e-4 * 64 * 5000))
    assert int((np.abs(x) == 30.0).sum()) == n
    t = d["targets"]
    assert t.dtype == np.int32 and t.min() >= 0 and t.max() < 5000
    assert d["grad_scale"] == 1.0 / 64


def test_router_quantised_ties_and_blocked_rows():
    d = inputs.router(0, rows=10000, cols=64)
    x, m = d["x"], d["mask"]
    assert np.array_equal(x * 8, np.round(x * 8)) and x.min() >= -4 and x.max() <= 4
    assert m.dtype == np.uint8 and set(np.unique(m)) <= {0, 1}
    assert len(d["blocked_rows"]) == 100
    assert not m[d["blocked_rows"]].any()
    live = np.setdiff1d(np.arange(10000), d["blocked_rows"])
    assert abs(m[live].mean() - 0.9) < 0.01


def test_attention_shape():
    d = inputs.attention(0, batch=1, heads=2, seq=64)
    assert d["scores"].shape == (128, 64) and d["seq_len"] == 64 and d["scale"] == 0.125
