"""The seeded input generator: bf16 rounding against torch, determinism, shapes."""
import numpy as np
import torch

from workloads import WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_activations, make_weights


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
