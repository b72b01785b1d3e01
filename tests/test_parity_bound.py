"""The per-element bound that the GPU parity tests apply to bf16 outputs (tests.gpu_util),
pinned against torch's bf16 rounding on the CPU."""


def test_parity_bound_for_bf16_outputs():
    """The per-element bound of the GPU parity tests: 1e-2, except where half a bf16 ulp of
    the exact value exceeds it (|x| >= 4), where the output must be faithfully rounded."""
    import numpy as np
    import torch

    from tests.gpu_util import allowed_error, bf16_ulp
    assert bf16_ulp(np.array([1.0, 1.5, 2.0, 4.55, -4.55, 0.25]))[[0, 1, 2, 3, 4, 5]].tolist() == \
        [2.0 ** -7, 2.0 ** -7, 2.0 ** -6, 2.0 ** -5, 2.0 ** -5, 2.0 ** -9]
    x = np.concatenate([np.linspace(-9, 9, 200001), [3.999, 4.0, 4.55, 7.9]])
    a = allowed_error(x, True)
    assert (a[np.abs(x) < 4] == 1e-2).all() and (a[np.abs(x) >= 4] > 1e-2).all()
    # every exact value rounded to bf16 (nearest even) passes; its next bf16 neighbour
    # further away fails wherever the bound is one ulp
    r = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert (np.abs(r - x) <= a).all()
    far = r + np.sign(r - x + 1e-300) * bf16_ulp(x)
    big = np.abs(x) >= 4
    assert (np.abs(far - x)[big] > a[big]).all()
    assert allowed_error(x, False).max() == 1e-2
