"""kda_attn_res (AttnRes depth mixing) on the GPU against the float64 oracle:
float32 and bf16 stacks, block counts from 1 to the maximum, widths from 8 to
8192 (some not a multiple of the CTA's 256 x 16-byte sweep), more rows than
the grid holds at once, and the argument checks."""
import numpy as np
import pytest
import torch

import gated_delta_rule_wise_gb300 as kda
import oracle
import workloads as W
from _gpu_helpers import DEV, rel_err

pytestmark = pytest.mark.gpu


def _case(nb, rows, D, dtype, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    V = (scale * rng.standard_normal((nb, rows, D))).astype(np.float32)
    w = (rng.standard_normal(D) / np.sqrt(D) * 4.0).astype(np.float32)
    if dtype == "bf16":
        V = W.round_bf16(V)
    return V, w


@pytest.mark.parametrize("nb,rows,D,dtype", [
    (1, 5, 64, "f32"), (9, 33, 1024, "f32"), (9, 40, 7168, "bf16"), (32, 7, 520, "bf16"),
    (13, 300, 2056, "bf16"), (8, 1, 8, "f32"), (1, 3, 1024, "bf16"), (10, 17, 4096, "bf16"),
    (9, 400, 2048, "bf16"), (3, 2, 8192, "bf16"), (11, 6, 7168, "bf16"), (4, 5, 1536, "bf16")])
def test_attn_res_matches_oracle(nb, rows, D, dtype):
    V, w = _case(nb, rows, D, dtype, seed=nb * 7 + D)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    Vd = torch.from_numpy(V).to(DEV).to(tdt)
    h = kda.attn_res(Vd, torch.from_numpy(w).to(DEV))
    torch.cuda.synchronize()
    ref = oracle.attn_res(V, w)
    tol = 1e-2 if dtype == "bf16" else 1e-5
    assert rel_err(h.float().cpu().numpy(), ref) <= tol


def test_attn_res_bench_size_sampled_rows():
    """The bench's case, 9 blocks x 4096 rows x 7168 (bf16), in the bench's
    launch: more rows than the grid (16 CTAs per SM), so CTAs take a second
    row (and prefetch it).  Checked on a seeded sample of rows, among them the
    first rows past the grid."""
    nb, rows, D = 9, 4096, 7168
    V, w = _case(nb, rows, D, "bf16", seed=97)
    h = kda.attn_res(torch.from_numpy(V).to(DEV).to(torch.bfloat16), torch.from_numpy(w).to(DEV))
    torch.cuda.synchronize()
    grid = torch.cuda.get_device_properties(0).multi_processor_count * 16
    rng = np.random.default_rng(3)
    sample = np.unique(np.concatenate([rng.choice(rows, 48, replace=False),
                                       [0, grid - 1, grid, grid + 1, rows - 1]]))
    ref = oracle.attn_res(V[:, sample], w)
    assert rel_err(h.float().cpu().numpy()[sample], ref) <= 1e-2


def test_attn_res_weights_follow_the_scores():
    """Block 3 of every row made dominant: h is (nearly) that block."""
    V, w = _case(6, 64, 256, "f32", seed=5)
    w = 50.0 * np.abs(w)
    V[3] = np.abs(V[3]) + 0.5
    Vd = torch.from_numpy(V).to(DEV)
    h = kda.attn_res(Vd, torch.from_numpy(w).to(DEV))
    torch.cuda.synchronize()
    assert np.allclose(h.cpu().numpy(), oracle.attn_res(V, w), rtol=1e-5, atol=1e-6)
    assert np.allclose(h.cpu().numpy(), V[3], atol=1e-3)


def test_attn_res_argument_checks():
    V = torch.zeros((33, 2, 64), device=DEV)
    w = torch.zeros(64, device=DEV)
    h = torch.empty((2, 64), device=DEV)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_attn_res(V, w, h)
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED  # more than 32 blocks
    V2 = torch.zeros((4, 2, 60), device=DEV)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_attn_res(V2, torch.zeros(60, device=DEV), torch.empty((2, 60), device=DEV))
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED  # D not a multiple of 8
    with pytest.raises(kda.KdaError) as e:
        kda.kda_attn_res(V[:4], w, h, eps=-1.0)
    assert e.value.status == kda.KDA_ERR_INVALID_ARG
