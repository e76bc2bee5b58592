"""The local parity checks used by the GPU tests have teeth: on CPU, a
planted error confined to one (request, head) or one node row -- too small to
move the whole tensor's relative Frobenius error past the bound -- must be
rejected, and rounding-level noise everywhere must pass."""
import numpy as np
import pytest

from conftest import assert_local_parity, rel_fro, row_errors, state_unit_errors, unit_errors


def _forest(seed=0, B=64, H=32, d=128):
    rng = np.random.default_rng(seed)
    sizes = rng.integers(8, 65, size=B)
    offsets = np.zeros(B + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(sizes)
    ref = rng.standard_normal((int(offsets[-1]), H, d))
    return offsets, ref, rng


def test_one_wrong_head_is_caught_though_the_tensor_norm_passes():
    offsets, ref, rng = _forest()
    got = ref.copy()
    b, h = 17, 5
    o, e = offsets[b], offsets[b + 1]
    got[o:e, h] += 0.05 * rng.standard_normal(got[o:e, h].shape)  # 5% off in one head
    assert rel_fro(got, ref) < 1e-2
    assert unit_errors(got, ref, offsets)[(b, h)] > 1e-2
    with pytest.raises(AssertionError, match=r"\(17, 5\)"):
        assert_local_parity("planted", "O", got, ref, offsets, 1e-2)


def test_one_wrong_node_row_is_caught():
    offsets, ref, _ = _forest(1)
    got = ref.copy()
    b, node, h = 40, 3, 7
    got[offsets[b] + node, h] *= -1.0  # one row with the wrong sign
    assert rel_fro(got, ref) < 1e-2
    err, req = row_errors(got, ref, offsets)
    assert req[offsets[b] + node] == b and err[offsets[b] + node, h] > 1.0
    with pytest.raises(AssertionError):
        assert_local_parity("planted", "U", got, ref, offsets, 1e-2)


def test_rounding_noise_passes_and_tiny_rows_use_the_tensor_scale():
    offsets, ref, rng = _forest(2, B=8, H=4)
    ref[offsets[3] + 1, 2] *= 1e-6  # a row the oracle makes nearly zero
    got = ref * (1 + 2e-3 * rng.standard_normal(ref.shape))
    got[offsets[3] + 1, 2] += 1e-4  # absolute error far below the tensor's scale
    assert_local_parity("noise", "O", got, ref, offsets, 1e-2)


def test_state_units():
    rng = np.random.default_rng(3)
    ref = rng.standard_normal((4, 3, 16, 16))
    got = ref.copy()
    got[2, 1] += 0.1
    errs = state_unit_errors(got, ref)
    assert max(errs, key=errs.get) == (2, 1)
