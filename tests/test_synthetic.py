"""The seeded input generators that feed both the oracle and the library: same seed, same bits;
the documented shapes, ranges and outlier structure; and the 27B-class step whose algorithmic
bytes the benchmark divides by."""
import numpy as np
import torch

import synthetic


def test_same_seed_same_bits_and_seeds_separate():
    w1, s1 = synthetic.weights(4, 130, 256, 7)
    w2, s2 = synthetic.weights(4, 130, 256, 7)
    assert torch.equal(w1, w2) and torch.equal(s1.view(torch.int16), s2.view(torch.int16))
    w3, _ = synthetic.weights(4, 130, 256, 8)
    assert not torch.equal(w1, w3)
    x1 = synthetic.activations(3, 512, 5)
    assert torch.equal(x1.view(torch.int16), synthetic.activations(3, 512, 5).view(torch.int16))
    assert not torch.equal(x1.view(torch.int16), synthetic.activations(3, 512, 6).view(torch.int16))
    assert synthetic.sub_seed(1, "a", 2) == synthetic.sub_seed(1, "a", 2)
    assert synthetic.sub_seed(1, "a", 2) != synthetic.sub_seed(1, "a", 3)
    assert 0 <= synthetic.sub_seed(123, "x") < 2 ** 63


def test_weight_shapes_codes_and_scales():
    for bits, (c, eps) in ((4, (0.02, 1e-3)), (6, (0.005, 1e-4))):
        N, K = 257, 1024
        w, s = synthetic.weights(bits, N, K, 11)
        assert w.dtype == torch.uint8 and tuple(w.shape) == (N, synthetic.canonical_row_bytes(bits, K))
        assert s.dtype == torch.float16 and tuple(s.shape) == (N, K // 128)
        sf = s.float().numpy()
        assert np.isfinite(sf).all()
        assert sf.min() >= eps * (1 - 2 ** -10) and sf.max() < c * 6 + eps  # |N(0,1)| below 6 at this size
        # uniform bytes: every byte value occurs, and the mean is near 127.5
        counts = np.bincount(w.numpy().ravel(), minlength=256)
        assert (counts > 0).all() and abs(w.numpy().mean() - 127.5) < 2.0
    assert synthetic.canonical_row_bytes(4, 5120) == 2560 and synthetic.canonical_row_bytes(6, 5120) == 3840


def test_activation_outlier_channels():
    K = 5120
    n_out = int(round(0.01 * K))
    # over 64 rows the outlier channels (x20) stand clear of the N(0,1) ones by their mean |x|
    x64 = synthetic.activations(64, K, 21).float()
    assert torch.isfinite(x64).all()
    col = x64.abs().mean(dim=0)
    out = col > 4.0
    assert int(out.sum()) == n_out and col[~out].max() < 1.5 and col[out].min() > 8.0
    # the channels depend on the seed and K only, so a 4-row draw has the same ones: elsewhere
    # every value is a plain N(0,1) draw
    x4 = synthetic.activations(4, K, 21).float()
    assert tuple(x4.shape) == (4, K) and x4[:, ~out].abs().max() < 8.0
    plain = synthetic.activations(4, K, 21, outliers=False).float()
    assert plain.abs().max() < 8.0


def test_prologue_inputs():
    g = synthetic.rmsnorm_weight(4096, 3)
    assert g.dtype == torch.bfloat16 and g.shape == (4096,) and abs(g.float().mean().item() - 1.0) < 0.02
    gu = synthetic.gate_up_output(2, 1024, 3)
    assert gu.dtype == torch.float32 and tuple(gu.shape) == (2, 2048) and abs(gu.std().item() - 2.0) < 0.1


def test_27b_step_linears_and_bytes():
    lin = synthetic.step_27b()
    assert len(lin) == 257 and lin[-1] == ("lm_head", 5120, 152064)
    kinds = [name.split(".")[-1] for name, _, _ in lin[:-1]]
    assert kinds == ["qkv", "o", "gate_up", "down"] * 64
    # packed int4 weights + fp16 group scales + bf16 activations of one row, per step
    total = sum(N * K // 2 + 2 * N * (K // 128) + 2 * K for _, K, N in lin)
    assert total == 11_305_601_024
