"""The seeded generators: storage formats round-trip and match torch's casts."""
import numpy as np
import torch

from sparse_attention_indexer_idx_gb300 import workloads as wl


def test_bf16_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 100
    ours = wl.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(wl.bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_e4m3_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(100000) * 100, rng.standard_normal(1000) * 1e-3,
                        np.array([0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 1.5 * 2 ** -9])])
    x = x.astype(np.float32)
    x = np.clip(x, -448, 448)
    ours = wl.f32_to_e4m3_bits(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    assert np.array_equal(wl.e4m3_bits_to_f32(ours), torch.from_numpy(x).to(torch.float8_e4m3fn).float().numpy())


def test_generators_are_seeded():
    a = wl.tiny_fp32()
    b = wl.tiny_fp32()
    assert np.array_equal(a.q, b.q) and np.array_equal(a.keys, b.keys)
    p = wl.ragged_fp8(M=4, H=4, D=16, L_min=10, L_max=20)
    assert p.keys.dtype == np.uint8 and p.key_scale.shape[0] == p.n_keys
    assert int(p.key_off[-1] + p.key_len[-1]) == p.n_keys
    assert np.abs(p.keys_f32()).max() <= 448


def test_bulk_casts_equal_the_reference_encoders():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(50000) * 60).astype(np.float32)
    assert np.array_equal(wl._bulk_bf16(x), wl.f32_to_bf16_bits(x))
    y = np.clip(x, -448, 448)
    assert np.array_equal(wl._bulk_e4m3(y), wl.f32_to_e4m3_bits(y))
