"""The L1 training demo (train_demo.train): with the L1 term the hidden density
falls while the loss falls; without it the density stays high. Every forward
and backward runs through the library."""
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from activation_sparse_transformer_tcgen05_gb300 import build as _build
    _build.build()
from activation_sparse_transformer_tcgen05_gb300 import train_demo  # noqa: E402


def test_l1_training_raises_sparsity_and_fits():
    kw = dict(steps=400, M=1024, d=256, F=1024, T=128, lr=2e-3, log_every=100, verbose=False)
    with_l1 = train_demo.train(lam=0.05, **kw)
    without = train_demo.train(lam=0.0, **kw)
    first, last = with_l1[0], with_l1[-1]
    assert first["density"] > 0.4                      # ReLU at zero bias: about half active
    assert last["loss"] < 0.02 * first["loss"]         # it learns the teacher
    assert last["density"] < 0.5 * first["density"]    # and the L1 term sparsifies h
    assert without[-1]["density"] > 2 * last["density"]
