"""GPU parity: scaled causal attention softmax forward and backward."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import check_bound, check_exact_zero, check_probs, gpu, host, softmax_bwd_bound
from row_wise_softmax_warp_gb300 import inputs

pytestmark = pytest.mark.gpu


def _upper(rows, seq):
    q = np.arange(rows) % seq
    return np.arange(seq)[None, :] > q[:, None]


@pytest.mark.parametrize("seq", [1, 2, 3, 5, 8, 31, 64, 100, 256, 516, 600, 768, 1020, 1024, 1028, 1500, 2048,
                                 3001, 4096])
@pytest.mark.parametrize("misalign", [False, True])
def test_attention_shapes(ro, seq, misalign):
    heads = 3 if seq <= 256 else 1
    a = inputs.attention(seq, batch=1, heads=heads, seq=seq)
    s, dp, scale = a["scores"], a["dp"], a["scale"]
    rows = s.shape[0]
    # Garbage above the diagonal must not be read: poison it with NaN.
    s = s.copy()
    s[_upper(rows, seq)] = np.nan
    p = ro.rowops_attn_softmax_fwd(gpu(s, misalign), seq_len=seq, scale=scale)
    ref = oracle.attn_softmax_forward(np.where(np.isnan(s), 0, s), seq, scale)
    got = host(p)
    check_probs(got, ref, f"attn fwd seq={seq}")
    check_exact_zero(got, _upper(rows, seq), "attn fwd upper triangle")
    p32 = ref.astype(np.float32)
    p_in = p32.copy()
    p_in[_upper(rows, seq)] = np.nan
    dp_in = dp.copy()
    dp_in[_upper(rows, seq)] = np.nan
    ds = host(ro.rowops_attn_softmax_bwd(gpu(p_in, misalign), gpu(dp_in, misalign), seq_len=seq,
                                         scale=scale))
    dref = oracle.attn_softmax_backward(p32, dp, seq, scale)
    check_bound(ds, dref, softmax_bwd_bound(p32, np.where(_upper(rows, seq), 0, dp), scale),
                f"attn bwd seq={seq}")
    check_exact_zero(ds, _upper(rows, seq), "attn bwd upper triangle")


def test_attention_scale_not_power_of_two(ro):
    a = inputs.attention(1, batch=2, heads=2, seq=128)
    scale = 0.1
    p = host(ro.rowops_attn_softmax_fwd(gpu(a["scores"]), seq_len=128, scale=scale))
    check_probs(p, oracle.attn_softmax_forward(a["scores"], 128, scale), "scale 0.1")


def test_attention_first_query_and_equal_scores(ro):
    s = np.full((64, 64), 3.0, np.float32)
    p = host(ro.rowops_attn_softmax_fwd(gpu(s), seq_len=64, scale=0.125))
    assert p[0, 0] == 1.0 and (p[0, 1:] == 0).all()
    i = np.arange(64)
    check_probs(p, np.where(i[None, :] <= i[:, None], 1.0 / (i[:, None] + 1.0), 0.0), "equal scores")


def test_attention_empty(ro):
    x = torch.empty((0, 64), device="cuda")
    assert ro.rowops_attn_softmax_fwd(x, seq_len=64, scale=0.125).shape == (0, 64)
