"""The seeded input recipe (CPU): the generators are deterministic per seed and
draw the distributions the workloads state."""
import numpy as np
import torch

from bit_gradient_compression_gb300 import workloads as wl


def test_seed_convention():
    assert wl.seed_for(100, 3, 5) == 3105


def test_layout_sizes():
    assert wl.layout_numel(wl.llama2_7b_layout()) == 6_738_415_616
    assert wl.layout_numel(wl.tinyllama_layout()) == 1_100_048_384
    assert wl.layout_numel(wl.mixtral_moe_layer_layout()) == 1_409_286_144
    names = [n for n, _ in wl.llama2_7b_layout()]
    assert names[0] == "embed" and names[-1] == "head" and len(names) == 1 + 32 * 9 + 2


def test_llm_law_is_deterministic_with_per_tensor_sigma():
    layout = [("a", 20000), ("b", 30000), ("c", 25000)]
    n = wl.layout_numel(layout)
    x = wl.fill_llm_grads(torch.empty(n), layout, 7)
    y = wl.fill_llm_grads(torch.empty(n), layout, 7)
    z = wl.fill_llm_grads(torch.empty(n), layout, 8)
    assert torch.equal(x, y) and not torch.equal(x, z)
    off = 0
    for _, k in layout:
        s = float(x[off:off + k].std())
        assert 0.9e-5 <= s <= 1.1e-2          # sigma = 10**U(-5, -2) per tensor
        off += k


def test_moe_law_zero_experts_and_heavy_tails():
    layout = [(f"e{e}.w1", 40000) for e in range(8)]
    x = wl.fill_moe_grads(torch.empty(8 * 40000), layout, 3)
    for e in range(8):
        part = x[e * 40000:(e + 1) * 40000]
        if e in (3, 7):
            assert torch.count_nonzero(part) == 0
        else:
            a = part.numpy().astype(np.float64) / 1e-3
            kurt = ((a - a.mean()) ** 4).mean() / a.var() ** 2
            assert kurt > 6.0                  # Student-t(3): far heavier tails than a normal (3)


def test_flat_outliers_rate():
    x = wl.fill_flat_normal(torch.empty(1 << 20), 5, outlier_p=1e-3)
    big = (x.abs() > 1e-3 * 8).float().mean().item()   # beyond 8 sigma only the x100 outliers remain
    assert 0.5e-3 < big < 1.5e-3
