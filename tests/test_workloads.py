"""The seeded input recipe (CPU): exact spike counts, determinism, the
reference configuration's shape and scaled row, and the mixture-of-experts
split with its forced empty and sub-block experts."""
import numpy as np
import torch

from mxfp8_block_scaled_mx_gb300 import workloads as W


def test_synth_matrix_has_the_exact_spike_count_and_is_seeded():
    x = W.synth_matrix((300, 200), 1e-3, 0.01, 50.0, 60.0, seed=5)
    assert x.dtype == torch.bfloat16 and x.shape == (300, 200)
    big = x.float().abs() >= 49.5                 # spikes, after the bf16 cast
    assert int(big.sum()) == round(0.01 * 300 * 200)
    assert float(x.float().abs()[big].max()) <= 60.5
    signs = torch.sign(x.float()[big])
    assert 0 < int((signs > 0).sum()) < int(big.sum())   # both signs occur
    assert torch.equal(x, W.synth_matrix((300, 200), 1e-3, 0.01, 50.0, 60.0, seed=5))
    assert not torch.equal(x, W.synth_matrix((300, 200), 1e-3, 0.01, 50.0, 60.0, seed=6))
    plain = W.synth_matrix((64, 64), 0.02, seed=1)
    assert float(plain.float().std()) < 0.03


def test_reference_configuration():
    x, w = W.pr1_reference()
    assert x.shape == (256, 512) and w.shape == (512, 256)
    spikes = x.float().abs() >= 199.0
    assert int(spikes[1:].sum()) + int((x[0].float().abs() >= 0.199).sum()) == 1311
    assert float(x[0].float().abs().max()) < 0.61          # row 0 scaled by 1e-3
    assert float(w.float().std()) < 0.03


def test_moe_split_has_the_forced_edge_experts():
    sizes = W.moe_group_sizes(65536, 64, seed=0)
    assert sizes.sum() == 65536 and len(sizes) == 64
    assert (sizes == 0).sum() >= 2 and (sizes == 1).sum() >= 1 and (sizes == 31).sum() >= 1
    assert sizes.max() > 10000                               # Zipf head
    assert np.array_equal(sizes, W.moe_group_sizes(65536, 64, seed=0))
    off = W.moe_offsets(sizes)
    assert off.dtype == np.int32 and off[0] == 0 and off[-1] == 65536
    assert (np.diff(off) >= 0).all()


def test_random_bits_cover_the_16_bit_range():
    r = W.random_bits16((256, 256), seed=3)
    assert r.dtype == torch.int16 and r.shape == (256, 256)
    u = r.to(torch.int32) & 0xFFFF
    assert int(u.min()) < 256 and int(u.max()) > 65535 - 256
    assert abs(float(u.float().mean()) - 32767.5) < 500
    assert torch.equal(r, W.random_bits16((256, 256), seed=3))
