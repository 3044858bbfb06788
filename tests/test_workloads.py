"""The seeded input generator: bf16 rounding against torch, determinism, shapes."""
import numpy as np
import torch

from workloads import WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_activations, make_weights, random_matrix


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 100,
                        (np.arange(1 << 16, dtype=np.uint32) << 16 | 0x8000).view(np.float32)])
    x = x[np.isfinite(x)]
    ours = f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_row_slices_match_full_draw_and_are_deterministic():
    g = WORKLOADS["vitl_nvfp4"].gemms[0]
    small = make_activations(g, rows=64)
    again = make_activations(g, rows=64)
    assert np.array_equal(small, again)
    g2 = WORKLOADS["vitb_fc1_mxfp8"].gemms[0]
    assert make_weights(g2).shape == (3072, 768)
    x = bf16_bits_to_f32(make_activations(g2, rows=256))
    # 4 outlier channels (0.5 % of 768) scaled x20
    col_rms = np.sqrt((x.astype(np.float64) ** 2).mean(axis=0))
    assert (col_rms > 5).sum() == 4


def test_massive_activation_recipe():
    """The massive-activation stress input: maximum exactly 1992 on a special token, rms about 9,
    the large values confined to the first 5 tokens of each 1024-token image."""
    x = bf16_bits_to_f32(random_matrix(2053, 512, seed=11, dist="massive")).astype(np.float64)
    assert np.abs(x).max() == 1992.0
    assert 8.5 < np.sqrt(np.mean(x * x)) < 12.0
    special = (np.arange(2053) % 1024) < 5
    assert np.abs(x[~special]).max() < 100.0
    assert (np.abs(x[special]) >= 500.0).sum() == 2 * special.sum()
