"""Pins for the oracle's AttnRes depth mixing ("22,580: From GPT-2 to Kimi K3"
(yichencityu.github.io), section 12): stack the block representations,
RMS-normalise them as keys, score each with the learned vector, softmax over
the block axis, mix the values.  Pinned by special cases with closed forms and
by torch's own rms_norm / softmax."""
import numpy as np
import torch

import oracle


def _data(rng, nb=5, rows=7, D=24):
    return rng.standard_normal((nb, rows, D)), rng.standard_normal(D)


def test_single_block_is_identity():
    V, w = _data(np.random.default_rng(1), nb=1)
    assert np.array_equal(oracle.attn_res(V, w), V[0])


def test_zero_query_is_the_mean_over_blocks():
    V, _ = _data(np.random.default_rng(2))
    assert np.allclose(oracle.attn_res(V, np.zeros(V.shape[-1])), V.mean(axis=0), rtol=1e-14,
                       atol=1e-14)


def test_scores_ignore_each_block_scale():
    """RMS-normalised keys (eps = 0 here, so exactly): scaling block n by
    c_n > 0 leaves the weights, so h = sum_n a_n c_n V_n with the weights of
    the unscaled blocks."""
    rng = np.random.default_rng(3)
    V, w = _data(rng)
    c = rng.uniform(0.5, 3.0, V.shape[0])
    K = V / np.sqrt((V ** 2).mean(-1, keepdims=True))
    a = np.exp(K @ w)
    a /= a.sum(0)
    h = oracle.attn_res(c[:, None, None] * V, w, eps=0.0)
    assert np.allclose(h, (a[..., None] * c[:, None, None] * V).sum(0), rtol=1e-12, atol=1e-14)


def test_dominant_score_selects_its_block():
    rng = np.random.default_rng(4)
    V, _ = _data(rng, nb=4, rows=3, D=16)
    w = 400.0 * V[2, 0] / np.linalg.norm(V[2, 0])  # row 0 strongly prefers block 2
    h = oracle.attn_res(V, w)
    assert np.allclose(h[0], V[2, 0], atol=1e-8)


def test_matches_torch_rms_norm_and_softmax():
    rng = np.random.default_rng(5)
    V, w = _data(rng, nb=9, rows=11, D=32)
    tV = torch.from_numpy(V)
    K = torch.nn.functional.rms_norm(tV, (V.shape[-1],), eps=1e-6)
    a = torch.softmax(torch.einsum("d,nrd->nr", torch.from_numpy(w), K), dim=0)
    ref = torch.einsum("nr,nrd->rd", a, tV).numpy()
    assert np.allclose(oracle.attn_res(V, w), ref, rtol=1e-12, atol=1e-13)
