"""Dense block-scaled GEMMs over several 128 x 256 output tiles: an odd number of row tiles,
ragged N and K, a bias and second-level scales, for W4A8, W8A8 and W4A4, against the
oracle."""
import numpy as np
import pytest
import torch

import synth
from oracle import qgemm as OQ
from qwtest import dense_w4a8, dev, qw, repack, u16_view

pytestmark = pytest.mark.gpu


def assert_parity(C, R, absum, what=""):
    ok, ratio, frob = OQ.check_bf16_result(C, R, absum)
    assert ok, f"{what}: worst |err|/bound = {ratio:.3g}, rel frob = {frob:.3g}"


@pytest.mark.parametrize("M,N,K", [(300, 264, 384), (130, 512, 256), (640, 1280, 1024),
                                   (257, 768, 96), (1000, 384, 2048)])
def test_w4a8_tiles(M, N, K):
    p = synth.w4a8_problem(M, N, K, cfg_id=1300 + M)
    C = dense_w4a8(p)
    R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], K)
    assert_parity(C, R, S, f"W4A8 tiles {M}x{N}x{K}")


def test_w4a8_tiles_bias_and_scale2():
    Q = qw()
    M, N, K = 384, 520, 512
    p = synth.w4a8_problem(M, N, K, cfg_id=1320, bias=True)
    d, wp, sp = repack(Q.QW_W_MXFP4_G32 | Q.QW_W_SCALE2, 1, N, K, p["w_canon"], p["s_canon"])
    rng = np.random.default_rng(1321)
    t = (2.0 ** rng.integers(-3, 4, N)).astype(np.float32)
    err = Q.new_error_flag()
    Q.qw_repack_scale2(d, dev(t), sp, err)
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    Q.qgemm_dense(d, wp, sp, Q.QW_A_MXFP8_G32, dev(p["A"]), dev(p["A_sf"]),
                  dev(p["bias"][0].view(np.int16)), C, M, None, 0, err)
    assert Q.qw_read_error(err) == 0
    R, S = OQ.w4a8_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], K)
    R2, S2 = OQ.apply_scale2(R, S, t, p["bias"][0])
    assert_parity(u16_view(C), R2, S2, "W4A8 tiles bias + scale2")


@pytest.mark.parametrize("M,N,K", [(300, 264, 384), (256, 512, 256)])
def test_w8a8_tiles(M, N, K):
    Q = qw()
    p = synth.w8a8_problem(M, N, K, cfg_id=1330 + M)
    C = dense_w4a8(p, wfmt=Q.QW_W_MXFP8_G32)
    R, S = OQ.gemm_w8a8(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0])
    assert_parity(C, R, S, f"W8A8 tiles {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(300, 264, 512), (256, 512, 256)])
def test_w4a4_tiles(M, N, K):
    Q = qw()
    p = synth.w4a4_problem(M, N, K, cfg_id=1340 + M)
    d, wp, sp = repack(Q.QW_W_NVFP4_G16, 1, N, K, p["w_canon"], p["s_canon"])
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_dense(d, wp, sp, Q.QW_A_NVFP4_G16, dev(p["A"]), dev(p["A_sf"]), None, C, M, None, 0,
                  err)
    assert Q.qw_read_error(err) == 0
    R, S = OQ.w4a4_from_canonical(p["A"], p["A_sf"], p["w_canon"][0], p["s_canon"][0], K)
    assert_parity(u16_view(C), R, S, f"W4A4 tiles {M}x{N}x{K}")
