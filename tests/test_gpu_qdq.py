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


def test_fake_qdq_large_group_many_blocks():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((1, 2048, 2048)).astype(np.float32)   # one 4M-element group
    x[0, 1234, 777] = 91.5
    y_ref, s_ref = oracle.qdq_groups(x, 2048, "e4m3")
    y, s = fake_qdq_e4m3(torch.from_numpy(x).cuda(), 2048)
    assert np.array_equal(_bits(s.cpu().numpy()), _bits(s_ref))
    assert np.array_equal(_bits(y.cpu().numpy()), _bits(y_ref))
