"""Host-side tests of the C ABI: the library loads without a GPU, exports every
symbol the header declares, and rejects invalid problems before any CUDA call."""
import ctypes
import os
import re

import pytest
import torch

from gated_delta_rule_54_gb300 import _lib
from gated_delta_rule_54_gb300._lib import GdnProblem

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "gdn_qdq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*[\w\s\*]+?\b(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_symbols_all_exported_and_bound():
    lib = _lib.load()
    declared = _declared_symbols()
    assert "gdn_chunk_fwd_qdq" in declared and "fake_qdq_int8" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(_lib.SIGNATURES)


def _problem(**kw):
    p = GdnProblem()
    p.B, p.T, p.Hk, p.Hv, p.Dk, p.Dv, p.N = 2, 300, 2, 4, 128, 128, 2
    p.cu_seqlens = None
    p.scale = 1.0
    p.state_mode, p.w_mode, p.block_v, p.chunk, p.dtype = 1, 1, 64, 64, 0
    p.solve, p.solve_degree, p.save_ctx = 0, 0, 1
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _validate(p):
    return _lib.load().gdn_validate(ctypes.byref(p))


def test_validate_accepts_supported_problems():
    assert _validate(_problem()) == 0
    assert _validate(_problem(Dk=64, Dv=64)) == 0
    assert _validate(_problem(state_mode=2, w_mode=1, Hv=8)) == 0
    assert _validate(_problem(state_mode=0, w_mode=0)) == 0
    assert _validate(_problem(B=1, N=5, cu_seqlens=4096)) == 0
    assert _validate(_problem(T=0)) == 0
    for bv in (16, 32, 128):
        assert _validate(_problem(block_v=bv)) == 0
    for deg in (0, 3, 63):
        assert _validate(_problem(solve=1, solve_degree=deg)) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=2), -2),                 # FP32 q/k/v rejected before launch
    (dict(dtype=1), -2),
    (dict(dtype=7), -1),
    (dict(Dk=96), -3), (dict(Dv=256), -3),
    (dict(Hv=3), -3),                    # Hv % Hk
    (dict(chunk=32), -3),
    (dict(block_v=48), -4), (dict(block_v=128, Dv=64), -4),
    (dict(solve=2), -1), (dict(solve=1, solve_degree=64), -4), (dict(solve=1, solve_degree=-1), -4),
    (dict(state_mode=3), -1), (dict(w_mode=-1), -1),
    (dict(B=-1), -1), (dict(Hk=0), -1),
    (dict(N=3), -1),                     # N != B without cu_seqlens
    (dict(B=2, N=2, cu_seqlens=4096), -1),  # packed needs B == 1
    (dict(scale=float("nan")), -1),
])
def test_validate_rejects(kw, code):
    assert _validate(_problem(**kw)) == code


def test_sizes():
    lib = _lib.load()
    p = _problem()
    nt = -(-300 // 64)
    assert lib.gdn_num_chunk_slots(ctypes.byref(p)) == 2 * nt
    al = lambda x: (x + 255) // 256 * 256
    ns = 2 * nt
    cv = al(4 * ns * 4 * 5 * 64)                                    # chunk vectors
    imgs = 3 * al(ns * 4 * 64 * 64 * 2) + al(ns * 4 * 2 * 64 * 64 * 2)  # T / GKK / P, Delta images
    imgs_tc = 2 * al(ns * 4 * 64 * 64 * 2)   # T / P: the tensor-core backward recomputes the others
    tf = al(4 * ns * 4 * 64 * 64)                                   # fp32 T of the fused forward
    w = al(2 * 300 * 4 * 128) + al(4 * ns * 4)                      # W codes and scales
    h = al(ns * 4 * 128 * 128) + al(4 * ns * 4 * 2)                 # state codes and scales
    # Dk = Dv = 128, both sites quantized, block_v 64: the fused forward
    assert lib.gdn_ctx_bytes(ctypes.byref(p)) == w + cv + imgs_tc + tf + h
    # forward only: no backward tiles; the fused forward keeps the states on chip
    assert lib.gdn_ctx_bytes(ctypes.byref(_problem(save_ctx=0))) == w + cv + tf
    # the three-launch path (here block_v 32) hands the state codes to its output pass
    h32 = al(ns * 4 * 128 * 128) + al(4 * ns * 4 * 4)
    assert lib.gdn_ctx_bytes(ctypes.byref(_problem(block_v=32, save_ctx=0))) == w + cv + h32
    p0 = _problem(state_mode=0, w_mode=0)
    assert lib.gdn_ctx_bytes(ctypes.byref(p0)) == al(4 * 2 * 300 * 4 * 128) + cv + imgs + al(4 * ns * 4 * 128 * 128)
    # segment offsets: the first is at 0, absent ones are -1, and they are increasing
    offs = [lib.gdn_ctx_offset(ctypes.byref(p), s) for s in range(12)]
    assert offs[0] == 0 and offs[2] == -1 and offs[11] == -1
    present = [o for o in offs if o >= 0]
    assert present == sorted(present) and len(present) == 8
    assert offs[5] == -1 and offs[7] == -1   # no Gamma o KK^T or Delta images
    po = _problem(save_ctx=0)
    assert [lib.gdn_ctx_offset(ctypes.byref(po), s) >= 0 for s in range(12)] == \
        [True, True, False, True, False, False, False, False, True, False, False, False]
    pk = _problem(B=1, T=1000, N=7, cu_seqlens=4096)
    assert lib.gdn_num_chunk_slots(ctypes.byref(pk)) == 1000 // 64 + 7
    assert lib.gdn_ctx_bytes(ctypes.byref(_problem(Dk=96))) == 0
    assert lib.gdn_num_chunk_slots(ctypes.byref(_problem(Dk=96))) == -1
    assert lib.gdn_ctx_offset(ctypes.byref(_problem(Dk=96)), 0) == -1
    assert _validate(_problem(save_ctx=2)) == -1


def test_packed_slot_formula_is_injective():
    # slot(n, c) = floor(cu[n]/64) + n + c never collides and stays below floor(T/64) + N
    import numpy as np
    rng = np.random.default_rng(0)
    for _ in range(200):
        lens = rng.integers(0, 300, rng.integers(1, 12))
        cu = np.concatenate([[0], np.cumsum(lens)])
        T, N = int(cu[-1]), len(lens)
        slots = [cu[n] // 64 + n + c for n in range(N) for c in range(-(-int(lens[n]) // 64))]
        assert len(set(slots)) == len(slots)
        assert all(0 <= s < T // 64 + N for s in slots)


def test_entry_points_reject_before_launch():
    lib = _lib.load()
    bad = _problem(dtype=2)
    P = ctypes.c_void_p
    fake = P(4096)
    assert lib.gdn_chunk_fwd_qdq(ctypes.byref(bad), fake, fake, fake, fake, fake, None, fake,
                                 None, None, None) == -2
    ok = _problem()
    # null inputs
    assert lib.gdn_chunk_fwd_qdq(ctypes.byref(ok), None, fake, fake, fake, fake, None, fake,
                                 None, None, None) == -1
    # misaligned pointer
    assert lib.gdn_chunk_fwd_qdq(ctypes.byref(ok), P(4097), fake, fake, fake, fake, None, fake,
                                 None, None, None) == -7
    # ctx must be 256-byte aligned, and is required
    assert lib.gdn_chunk_fwd_qdq(ctypes.byref(ok), fake, fake, fake, fake, fake, None, fake,
                                 None, P(4096 + 16), None) == -7
    assert lib.gdn_chunk_fwd_qdq(ctypes.byref(ok), fake, fake, fake, fake, fake, None, fake,
                                 None, None, None) == -1
    # backward: workspace too small
    need = lib.gdn_bwd_workspace_bytes(ctypes.byref(ok))
    if need > 0:
        args = [fake] * 14
        st = lib.gdn_chunk_bwd_ste(ctypes.byref(ok), *args[:6], fake, None, *[fake] * 5, None,
                                   fake, ctypes.c_size_t(need - 1), None)
        assert st == -5
    # fake QDQ argument checks
    assert lib.fake_qdq_e4m3(fake, fake, fake, None, 1, 4, 100, 64, None) == -1   # 100 % 64
    assert lib.fake_qdq_int8(fake, fake, None, None, 1, 4, 128, 64, None) == -1   # scales required
    assert lib.fake_qdq_int8(P(4098), fake, fake, None, 1, 4, 128, 64, None) == -7
    assert lib.fake_qdq_e4m3(None, None, None, None, 0, 4, 128, 64, None) == 0     # empty


def test_status_strings():
    lib = _lib.load()
    for code in range(-7, 1):
        s = lib.gdn_status_string(code).decode()
        assert s.startswith("GDN_")
    assert lib.gdn_abi_version() == 7


def _dproblem(**kw):
    p = _lib.GdnDecodeProblem()
    p.B, p.T, p.Hk, p.Hv, p.Dk, p.Dv = 8, 1, 2, 4, 128, 128
    p.scale, p.state_mode, p.block_v, p.readout, p.dtype = 1.0, 1, 64, 0, 0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,code", [
    (dict(), 0), (dict(block_v=16), 0), (dict(block_v=32, Dv=64), 0), (dict(block_v=128), 0),
    (dict(state_mode=2, readout=1), 0), (dict(state_mode=0, T=0), 0), (dict(Dk=64, Dv=64), 0),
    (dict(dtype=2), -2), (dict(dtype=9), -1), (dict(Dk=96), -3), (dict(Hv=3), -3),
    (dict(block_v=128, Dv=64), -4), (dict(block_v=48), -4), (dict(block_v=8), -4),
    (dict(readout=2), -1), (dict(state_mode=3), -1), (dict(B=-1), -1), (dict(T=-1), -1),
    (dict(B=65536), -3), (dict(scale=float("nan")), -1),
])
def test_decode_validate(kw, code):
    assert _lib.load().gdn_decode_validate(ctypes.byref(_dproblem(**kw))) == code


def test_decode_entry_rejects_before_launch():
    lib = _lib.load()
    P = ctypes.c_void_p
    f = P(4096)
    ok = _dproblem()
    call = lambda p, *a: lib.gdn_decode_qdq(ctypes.byref(p), *a)
    assert call(_dproblem(dtype=2), f, f, f, f, f, f, f, f, None, None, None) == -2
    assert call(ok, None, f, f, f, f, f, f, f, None, None, None) == -1          # null q
    assert call(ok, f, f, f, f, f, f, f, None, None, None, None) == -1          # null state_out
    assert call(ok, P(4100), f, f, f, f, f, f, f, None, None, None) == -7       # misaligned
    # state_out overlapping state_in without being it
    n = 8 * 4 * 128 * 128 * 4
    assert call(ok, f, f, f, f, f, P(1 << 20), f, P((1 << 20) + n // 2), None, None, None) == -1
    assert call(_dproblem(B=0), None, None, None, None, None, None, None, None, None, None,
                None) == 0


def _tproblem(**kw):
    p = _lib.GdnTwoPrecisionProblem()
    p.B, p.T, p.Hk, p.Hv, p.Dk, p.Dv, p.N = 2, 100, 2, 4, 128, 128, 2
    p.scale, p.read_mode, p.flush, p.dtype = 1.0, 1, 16, 0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,code", [
    (dict(), 0), (dict(read_mode=0), 0), (dict(Dv=64), 0), (dict(flush=1), 0), (dict(T=0), 0),
    (dict(flush=100000), 0), (dict(read_mode=2), -4), (dict(read_mode=7), -1), (dict(flush=0), -1),
    (dict(Dk=64), -3), (dict(Dv=96), -3), (dict(Hv=3), -3), (dict(dtype=2), -2), (dict(dtype=1), -2),
    (dict(N=3), -1), (dict(B=-1), -1), (dict(scale=float("nan")), -1),
    (dict(B=70000, N=70000), -3),
])
def test_two_precision_validate(kw, code):
    assert _lib.load().gdn_two_precision_validate(ctypes.byref(_tproblem(**kw))) == code


def test_two_precision_entry_rejects_before_launch():
    lib = _lib.load()
    P = ctypes.c_void_p
    f = P(4096)
    call = lambda p, *a: lib.gdn_two_precision_fwd(ctypes.byref(p), *a)
    assert call(_tproblem(read_mode=2), f, f, f, f, f, None, f, f, None, None) == -4
    assert call(_tproblem(), None, f, f, f, f, None, f, f, None, None) == -1          # null q
    assert call(_tproblem(), f, f, f, f, f, None, None, f, None, None) == -1          # null o
    assert call(_tproblem(), f, f, f, f, f, P(4104), f, f, None, None) == -7          # misaligned h0
    assert call(_tproblem(), f, f, f, f, f, None, f, f, P(4100), None) == -7          # misaligned anchors
    # packed sequences: B == 1 and N >= 1
    assert lib.gdn_two_precision_validate(ctypes.byref(_tproblem(B=2, N=3, cu_seqlens=f))) == -1
    assert lib.gdn_two_precision_validate(ctypes.byref(_tproblem(B=1, N=3, cu_seqlens=f))) == 0
    # nothing to do: no sequences, or no tokens and no final state
    assert call(_tproblem(B=0, N=0), None, None, None, None, None, None, None, None, None, None) == 0
    assert call(_tproblem(T=0), None, None, None, None, None, None, None, None, None, None) == 0


def test_two_precision_anchor_and_workspace_sizes():
    lib = _lib.load()
    p = _tproblem()
    nwin = p.B * p.T // p.flush + p.N        # an anchor [Hv, 128, Dv] per window slot
    assert lib.gdn_two_precision_anchor_bytes(ctypes.byref(p)) == nwin * p.Hv * 128 * p.Dv * 4
    assert lib.gdn_two_precision_anchor_bytes(ctypes.byref(_tproblem(read_mode=2))) == 0
    assert lib.gdn_two_precision_bwd_workspace_bytes(ctypes.byref(p)) > 0
    # grouped heads add the per-value-head dq and dk
    g1 = lib.gdn_two_precision_bwd_workspace_bytes(ctypes.byref(_tproblem(Hk=4, Hv=4)))
    g2 = lib.gdn_two_precision_bwd_workspace_bytes(ctypes.byref(_tproblem(Hk=2, Hv=4)))
    assert g2 >= g1 + 2 * p.B * p.T * 4 * 128 * 4
    # windows longer than 256 tokens (and than the sequence) are not replayed
    assert lib.gdn_two_precision_bwd_workspace_bytes(ctypes.byref(_tproblem(T=1000, flush=300))) == 0
    assert lib.gdn_two_precision_bwd_workspace_bytes(ctypes.byref(_tproblem(T=200, flush=300))) > 0


def test_two_precision_bwd_rejects_before_launch():
    lib = _lib.load()
    P = ctypes.c_void_p
    f = P(4096)
    ws_ok = lib.gdn_two_precision_bwd_workspace_bytes(ctypes.byref(_tproblem()))

    def call(p, q=f, anchors=f, dO=f, dq=f, dht=None, ws=f, ws_bytes=ws_ok):
        return lib.gdn_two_precision_bwd(ctypes.byref(p), q, f, f, f, f, anchors, dO, dht, dq, f, f,
                                         f, f, None, ws, ws_bytes, None)
    assert call(_tproblem(read_mode=2)) == -4
    assert call(_tproblem(T=1000, flush=300)) == -3
    assert call(_tproblem(), q=None) == -1
    assert call(_tproblem(), anchors=None) == -1       # the forward's anchors are required
    assert call(_tproblem(), dO=None) == -1
    assert call(_tproblem(), dq=P(4100)) == -7
    assert call(_tproblem(), dht=P(4104)) == -7
    assert call(_tproblem(), ws_bytes=ws_ok - 1) == -5
    assert call(_tproblem(), ws=None) == -5
    assert call(_tproblem(B=0, N=0), q=None, anchors=None, dO=None, dq=None, ws=None, ws_bytes=0) == 0


def test_no_host_fallback_for_cpu_tensors():
    """Every compute entry point of the binding refuses host tensors: there is no
    CPU path behind the library."""
    from gated_delta_rule_54_gb300 import (gdn_chunk_fwd_qdq, gdn_decode_qdq, gdn_two_precision_bwd,
                                           gdn_two_precision_fwd, kda_recurrent_fwd_qdq,
                                           fake_qdq_e4m3, synth)
    d = synth.make_inputs(synth.small(B=1, T=8, Hk=1, Hv=1, Dk=64, Dv=64, h0=True, seed=1))
    with pytest.raises(ValueError, match="CUDA tensor"):
        gdn_chunk_fwd_qdq(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    with pytest.raises(ValueError, match="CUDA tensor"):
        gdn_decode_qdq(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    with pytest.raises(ValueError, match="CUDA tensor"):
        gdn_two_precision_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    with pytest.raises(ValueError, match="CUDA tensor"):
        gdn_two_precision_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                              torch.zeros(d["v"].shape))
    gk = d["g"][..., None].expand(*d["g"].shape, 64).contiguous()
    with pytest.raises(ValueError, match="CUDA tensor"):
        kda_recurrent_fwd_qdq(d["q"], d["k"], d["v"], d["beta"], gk, d["h0"])
    with pytest.raises(ValueError, match="CUDA float32 tensor"):
        fake_qdq_e4m3(torch.zeros(1, 4, 64), 64)
