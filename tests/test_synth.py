"""The seeded input generators: determinism, ranges and the post-pass."""
import torch

from int_tensor_reductions_gb300 import synth


def test_uniform_range_and_no_zeros():
    x = synth.uniform((1 << 16,), -1.0, 1.0, 0)
    assert x.dtype == torch.float32
    assert float(x.min()) >= -1.0 and float(x.max()) < 1.0
    assert int((x == 0).sum()) == 0
    assert int(((x.abs() < synth.FLT_MIN)).sum()) == 0


def test_seed_determinism():
    a = synth.normal((1000,), 1)
    b = synth.normal((1000,), 1)
    c = synth.normal((1000,), 2)
    assert torch.equal(a, b)
    assert not torch.equal(a, c)


def test_post_pass_replaces_zeros_and_denormals():
    x = torch.tensor([0.0, -0.0, 1e-40, -1e-40, 1.0, -2.0], dtype=torch.float32)
    synth._post(x)
    assert x.tolist() == [synth.TINY, synth.TINY, synth.TINY, synth.TINY, 1.0, -2.0]


def test_ragged_offsets_lengths():
    off = synth.ragged_offsets(5000, 8, 40, 5)
    lens = off[1:] - off[:-1]
    assert off.dtype == torch.int64 and int(off[0]) == 0
    assert int(lens.min()) == 8 and int(lens.max()) == 40
    x, off2 = synth.cfg5(rows=3000)
    assert x.numel() == int(off2[-1])
    assert float(x.min()) >= -4.0 and float(x.max()) < 4.0


def test_int_choice_values():
    x = synth.cfg4b(R=8, C=1024)
    assert x.dtype == torch.int32
    assert set(torch.unique(x).tolist()) == set(synth.INT_CHOICES)


def test_cfg_shapes_small():
    x, dst = synth.cfg2(rows=16, length=32)
    assert x.shape == (16, 32) and dst.shape == (16,)
    assert synth.cfg4a(R=4, C=8).shape == (4, 8)
    assert synth.cfg1(n=100).shape == (100,)
    v = synth.cfg4a(R=64, C=64)
    assert float(v.min()) >= 0.999 and float(v.max()) <= 1.001
