"""GPU: the standalone fake QDQ kernels are bit-exact with the oracle's fp32 QDQ."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_54_gb300 import fake_qdq_e4m3, fake_qdq_int8

pytestmark = pytest.mark.gpu

FN = {"e4m3": fake_qdq_e4m3, "int8": fake_qdq_int8}


def _bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("mode", ["e4m3", "int8"])
@pytest.mark.parametrize("shape,gc", [((5, 128, 128), 64), ((1, 1, 4096), 4096), ((3, 7, 96), 32),
                                      ((2, 64, 128), 128), ((1, 300, 64), 64)])
def test_fake_qdq_bit_exact(mode, shape, gc):
    rng = np.random.default_rng(zlib.crc32(repr((mode, shape, gc)).encode()))
    x = (rng.standard_normal(shape) * np.exp(rng.uniform(-8, 8, (shape[0], 1, 1)))).astype(np.float32)
    x[..., 0, :3] = [0.0, -0.0, -1e-30]
    y_ref, s_ref, c_ref = oracle.qdq_groups(x, gc, mode, with_codes=True)
    y, s, c = FN[mode](torch.from_numpy(x).cuda(), gc, with_codes=True)
    assert np.array_equal(_bits(s.cpu().numpy()), _bits(s_ref))
    assert np.array_equal(c.cpu().numpy(), c_ref)
    assert np.array_equal(_bits(y.cpu().numpy()), _bits(y_ref))


@pytest.mark.parametrize("mode", ["e4m3", "int8"])
def test_fake_qdq_zero_group_and_in_place(mode):
    x = np.zeros((2, 8, 64), np.float32)
    x[1] = np.linspace(-3, 5, 512, dtype=np.float32).reshape(8, 64)
    x[0, 2, 5] = -0.0
    y_ref, s_ref, c_ref = oracle.qdq_groups(x, 64, mode, with_codes=True)
    xt = torch.from_numpy(x).cuda()
    y, s, c = FN[mode](xt, 64, with_codes=True, out=xt)   # y aliases x
    assert y.data_ptr() == xt.data_ptr()
    assert np.array_equal(_bits(xt.cpu().numpy()), _bits(y_ref))
    assert np.array_equal(c.cpu().numpy(), c_ref)
    assert s.cpu().numpy()[0, 0] == 0.0


@pytest.mark.parametrize("mode", ["e4m3", "int8"])
def test_fake_qdq_tiny_amax_groups(mode):
    """Groups whose amax sits around the point where fl(1/s) overflows, with
    zeros inside: bit-exact with the oracle, and finite."""
    M = 448.0 if mode == "e4m3" else 127.0
    amax = [M * 2.0 ** -126, M * 2.0 ** -127, M * 2.0 ** -128, M * 2.0 ** -129, 1e-40, 2.0 ** -149]
    rng = np.random.default_rng(12)
    x = rng.uniform(-1, 1, (len(amax), 16, 64)).astype(np.float32)
    for b, a in enumerate(amax):
        x[b] *= np.float32(a) / np.abs(x[b]).max()
        x[b, 0, 0] = np.float32(a)
        x[b, 3, :4] = [0.0, -0.0, 0.0, -0.0]
    y_ref, s_ref, c_ref = oracle.qdq_groups(x, 64, mode, with_codes=True)
    y, s, c = FN[mode](torch.from_numpy(x).cuda(), 64, with_codes=True)
    y = y.cpu().numpy()
    assert np.isfinite(y).all()
    assert np.array_equal(_bits(s.cpu().numpy()), _bits(s_ref))
    assert np.array_equal(c.cpu().numpy(), c_ref)
    assert np.array_equal(_bits(y), _bits(y_ref))


def test_fake_qdq_large_group_many_blocks():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((1, 2048, 2048)).astype(np.float32)   # one 4M-element group
    x[0, 1234, 777] = 91.5
    y_ref, s_ref = oracle.qdq_groups(x, 2048, "e4m3")
    y, s = fake_qdq_e4m3(torch.from_numpy(x).cuda(), 2048)
    assert np.array_equal(_bits(s.cpu().numpy()), _bits(s_ref))
    assert np.array_equal(_bits(y.cpu().numpy()), _bits(y_ref))
