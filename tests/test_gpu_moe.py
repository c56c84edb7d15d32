"""MoE routing (bit-exact) and grouped GEMM parity on the GPU against the oracle."""
import functools

import numpy as np
import pytest
import torch

import synth
from oracle import moe as OM
from oracle import qgemm as OQ
from oracle import formats as OF
from qwtest import dev, host, qw, repack, route, u16_view

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,E,k", [(4096, 256, 8), (1, 128, 8), (16, 128, 8), (256, 128, 8),
                                   (2048, 128, 8), (8192, 128, 8), (3, 6, 3), (100, 1000, 32),
                                   (0, 64, 4), (7, 33, 1)])
def test_route_bit_exact(T, E, k):
    logits = synth.router_logits(T, E, cfg_id=3)
    ids, sp, off = route(logits, k)
    rids, rcounts, roff, rsp = OM.route(logits, k)
    assert np.array_equal(ids, rids)
    assert np.array_equal(off, roff)
    assert np.array_equal(sp, rsp)


def test_route_ties_bit_exact():
    rng = np.random.default_rng(9)
    logits = rng.integers(-2, 3, (300, 40)).astype(np.float32)  # heavy ties
    ids, sp, off = route(logits, 6)
    rids, _, roff, rsp = OM.route(logits, 6)
    assert np.array_equal(ids, rids) and np.array_equal(off, roff) and np.array_equal(sp, rsp)


@functools.lru_cache(maxsize=4)
def _weights(kind, E, N, K, bits, cfg_id):
    if kind == "mx":
        return synth.w4a8_problem(1, N, K, E=E, cfg_id=cfg_id)
    return synth.w4a16_problem(1, N, K, bits=bits, E=E, cfg_id=cfg_id)


def run_moe(afmt, wfmt, E, T, K, N, topk, cfg_id, bits=4, indexed=False):
    """Route -> permute -> grouped GEMM through the C ABI.  Returns host arrays (and, with
    ``indexed``, also the output of the indexed call on the unpermuted activations)."""
    Q = qw()
    logits = synth.router_logits(T, E, cfg_id=cfg_id)
    kind = "mx" if wfmt == Q.QW_W_MXFP4_G32 else "int"
    w = _weights(kind, E, N, K, bits, cfg_id)
    if kind == "mx":
        a = synth.w4a8_problem(T, 32, K, cfg_id=cfg_id + 1000)
        p = dict(w, A=a["A"], A_sf=a["A_sf"])
    else:
        a = synth.w4a16_problem(T, 16, K, cfg_id=cfg_id + 1000)
        p = dict(w, A=a["A"])
    d, wp, sp_ = repack(wfmt, E, N, K, p["w_canon"], p["s_canon"])
    P = T * topk
    lg = dev(logits)
    ids = torch.empty((T, topk), dtype=torch.int32, device="cuda")
    sp = torch.empty((P,), dtype=torch.int32, device="cuda")
    off = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
    n = Q.qgemm_moe_route_workspace_size(T, E, topk)
    rws = torch.empty(n, dtype=torch.uint8, device="cuda")
    Q.qgemm_moe_route(lg, T, E, topk, ids, sp, off, rws, n)
    if afmt == Q.QW_A_BF16:
        A = dev(p["A"].view(np.int16))
        As = torch.empty((P, K), dtype=torch.int16, device="cuda")
        Q.qgemm_moe_permute(afmt, A, None, K, sp, P, topk, As, None)
        Asf_s = None
    else:
        A = dev(p["A"])
        Asf = dev(p["A_sf"])
        As = torch.empty((P, K), dtype=torch.uint8, device="cuda")
        Asf_s = torch.empty((P, K // 32), dtype=torch.uint8, device="cuda")
        Q.qgemm_moe_permute(afmt, A, Asf, K, sp, P, topk, As, Asf_s)
    C = torch.full((P, N), -1, dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, afmt, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_grouped(d, wp, sp_, afmt, As, Asf_s, off, P, None, C, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    if not indexed:
        return p, logits, host(sp), host(off), u16_view(C)
    Ci = torch.full((P, N), -1, dtype=torch.int16, device="cuda")
    Q.qgemm_moe_grouped_indexed(d, wp, sp_, afmt, A, Asf, T, sp, topk, off, P, None, Ci, ws, wsn,
                                err)
    assert Q.qw_read_error(err) == 0
    return p, logits, host(sp), host(off), u16_view(C), u16_view(Ci)


@pytest.mark.parametrize("E,T,K,N", [(8, 40, 256, 384), (16, 64, 512, 512), (32, 300, 128, 640)])
def test_moe_grouped_w4a8_small(E, T, K, N):
    Q = qw()
    p, logits, sp, off, C = run_moe(Q.QW_A_MXFP8_G32, Q.QW_W_MXFP4_G32, E, T, K, N, 8, 300 + E)
    _, _, roff, rsp = OM.route(logits, 8)
    assert np.array_equal(off, roff) and np.array_equal(sp, rsp)
    tok = rsp // 8
    codes = OF.unpack_e2m1_bytes(p["w_canon"], K)
    R, S = OM.grouped_w4a8(p["A"][tok], p["A_sf"][tok], roff, codes, p["s_canon"])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("E,T,K,N,topk", [(8, 40, 256, 384, 8), (16, 300, 640, 256, 2),
                                          (32, 129, 128, 640, 4), (4, 3, 96, 256, 1)])
def test_moe_grouped_indexed_w4a8_equals_permute_then_grouped(E, T, K, N, topk):
    """The Indexed path (rows gathered by pair id inside the kernel, TMA gather4) gives the
    permuted path's output bit for bit, and both match the oracle."""
    Q = qw()
    p, logits, sp, off, C, Ci = run_moe(Q.QW_A_MXFP8_G32, Q.QW_W_MXFP4_G32, E, T, K, N, topk,
                                        310 + E, indexed=True)
    assert np.array_equal(C, Ci), f"{np.sum(C != Ci)} of {C.size} differ"
    _, _, roff, rsp = OM.route(logits, topk)
    tok = rsp // topk
    codes = OF.unpack_e2m1_bytes(p["w_canon"], K)
    R, S = OM.grouped_w4a8(p["A"][tok], p["A_sf"][tok], roff, codes, p["s_canon"])
    ok, ratio, frob = OQ.check_bf16_result(Ci, R, S)
    assert ok, (ratio, frob)


def test_moe_grouped_indexed_flags_bad_pairs():
    """A pair id outside [0, T*topk) is reported through the device error flag (its row
    reads token 0) instead of being followed out of bounds."""
    Q = qw()
    E, T, K, N, topk = 4, 16, 128, 256, 2
    w = _weights("mx", E, N, K, 4, 330)
    a = synth.w4a8_problem(T, 32, K, cfg_id=331)
    d, wp, spk = repack(Q.QW_W_MXFP4_G32, E, N, K, w["w_canon"], w["s_canon"])
    P = T * topk
    pairs = np.arange(P, dtype=np.int32)
    pairs[5] = P + 7
    off = np.array([0, 8, 16, 24, 32], dtype=np.int32)
    C = torch.zeros((P, N), dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_MXFP8_G32, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_grouped_indexed(d, wp, spk, Q.QW_A_MXFP8_G32, dev(a["A"]), dev(a["A_sf"]), T,
                                dev(pairs), topk, dev(off), P, None, C, ws, wsn, err)
    assert Q.qw_read_error(err) == Q.QW_ERR_INVALID_ARG


@pytest.mark.parametrize("T", [1, 16, 64])
@pytest.mark.parametrize("bits", [4, 3, 2])
def test_moe_grouped_w4a16_small_t(T, bits):
    """E=128 top-8, intermediate 640: up-projection K=4096 -> N=1280 (gate+up)."""
    Q = qw()
    p, logits, sp, off, C = run_moe(Q.QW_A_BF16, {4: 0, 3: 1, 2: 6}[bits], 128, T, 4096, 1280, 8,
                                    4, bits=bits)
    _, _, roff, rsp = OM.route(logits, 8)
    tok = rsp // 8
    q = {4: OF.unpack_int4, 3: OF.unpack_int3, 2: OF.unpack_int2}[bits](p["w_canon"], 4096)
    R, S = OM.grouped_w4a16(p["A"][tok], roff, q, p["s_canon"])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("T", [12, 32])
def test_moe_grouped_w4a16_around_the_path_switch(T):
    """E=8 top-8: 12 rows per expert (GEMV, two 8-row slices per tile) and 32 rows per
    expert (tcgen05 path); K=1024 -> N=512."""
    Q = qw()
    p, logits, sp, off, C = run_moe(Q.QW_A_BF16, 0, 8, T, 1024, 512, 8, 5)
    _, _, roff, rsp = OM.route(logits, 8)
    assert np.array_equal(off, roff) and np.array_equal(sp, rsp)
    R, S = OM.grouped_w4a16(p["A"][rsp // 8], roff, OF.unpack_int4(p["w_canon"], 1024),
                            p["s_canon"])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("T", [12, 32])
@pytest.mark.parametrize("bits", [4, 3, 2])
def test_moe_grouped_w4a16_ragged_n(T, bits):
    """N = 264 (a 16-row block and a 128-row tile end inside the matrix; an expert's scale
    plane, G * N_pad BF16, is not a multiple of 256 bytes, so experts sit at the
    descriptor's rounded stride): every expert, through the GEMV and the tcgen05 path."""
    Q = qw()
    p, logits, sp, off, C = run_moe(Q.QW_A_BF16, {4: 0, 3: 1, 2: 6}[bits], 8, T, 512, 264, 8,
                                    6 + bits, bits=bits)
    _, _, roff, rsp = OM.route(logits, 8)
    q = {4: OF.unpack_int4, 3: OF.unpack_int3, 2: OF.unpack_int2}[bits](p["w_canon"], 512)
    R, S = OM.grouped_w4a16(p["A"][rsp // 8], roff, q, p["s_canon"])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


def test_moe_grouped_w4a16_down_k640():
    """Down-projection K=640 -> N=4096 (K not a multiple of 256) on a per-pair input."""
    Q = qw()
    p, logits, sp, off, C = run_moe(Q.QW_A_BF16, 0, 128, 16, 640, 4096, 8, 4)
    _, _, roff, rsp = OM.route(logits, 8)
    R, S = OM.grouped_w4a16(p["A"][rsp // 8], roff, OF.unpack_int4(p["w_canon"], 640),
                            p["s_canon"])
    ok, ratio, frob = OQ.check_bf16_result(C, R, S)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("bad", ["decreasing", "past_end", "negative"])
def test_grouped_rejects_bad_device_offsets(bad):
    """Offsets live in device memory, so the host cannot check them: the device tile-queue
    builder reports them (QW_ERR_INVALID_ARG) and schedules no tile for the bad segment."""
    Q = qw()
    E, P, K, N = 4, 64, 128, 64
    p = synth.w4a16_problem(P, N, K, bits=4, E=E, cfg_id=77)
    d, wp, sp_ = repack(Q.QW_W_INT4_G128_BF16, E, N, K, p["w_canon"], p["s_canon"])
    offs = {"decreasing": [0, 40, 20, 50, 64], "past_end": [0, 16, 32, 48, 100000],
            "negative": [-1000, 16, 32, 48, 64]}[bad]
    off = torch.tensor(offs, dtype=torch.int32, device="cuda")
    A = dev(p["A"].view(np.int16))
    C = torch.full((P, N), 0x7FC0, dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_BF16, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_grouped(d, wp, sp_, Q.QW_A_BF16, A, None, off, P, None, C, ws, wsn, err)
    assert Q.qw_read_error(err) == Q.QW_ERR_INVALID_ARG
    assert float((torch.ones(2, device="cuda") * 3).sum()) == 6.0  # context still usable


@pytest.mark.parametrize("T", [1, 16])
def test_grouped_gemv_reads_the_tile_queue_of_this_call(T):
    """The grouped GEMV starts as a programmatic dependent of the kernel that builds its
    tile queue in the workspace: it must read the queue (its tile count included) only
    after waiting for that kernel.  The workspace is zeroed before every call (a stale
    count of 0 would schedule no tile) and C is filled with NaN, so a row the kernel never
    wrote shows up; every row must match the oracle on each of several calls."""
    Q = qw()
    E, K, N, topk = 128, 4096, 1280, 8
    w = _weights("int", E, N, K, 4, 4)
    a = synth.w4a16_problem(T, 16, K, cfg_id=1004)
    logits = synth.router_logits(T, E, cfg_id=4)
    d, wp, sp_ = repack(Q.QW_W_INT4_G128_BF16, E, N, K, w["w_canon"], w["s_canon"])
    P = T * topk
    ids = torch.empty((T, topk), dtype=torch.int32, device="cuda")
    sp = torch.empty((P,), dtype=torch.int32, device="cuda")
    off = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
    n = Q.qgemm_moe_route_workspace_size(T, E, topk)
    rws = torch.empty(n, dtype=torch.uint8, device="cuda")
    A = dev(a["A"].view(np.int16))
    As = torch.empty((P, K), dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_BF16, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    C = torch.empty((P, N), dtype=torch.int16, device="cuda")
    err = Q.new_error_flag()
    _, _, roff, rsp = OM.route(logits, topk)
    R, S = OM.grouped_w4a16(a["A"][rsp // topk], roff, OF.unpack_int4(w["w_canon"], K),
                            w["s_canon"])
    lg = dev(logits)
    for _ in range(4):
        ws.zero_()
        C.fill_(0x7FC0)  # BF16 NaN
        Q.qgemm_moe_route(lg, T, E, topk, ids, sp, off, rws, n)
        Q.qgemm_moe_permute(Q.QW_A_BF16, A, None, K, sp, P, topk, As, None)
        Q.qgemm_moe_grouped(d, wp, sp_, Q.QW_A_BF16, As, None, off, P, None, C, ws, wsn, err)
        assert Q.qw_read_error(err) == 0
        got = u16_view(C)
        assert not np.any(got == 0x7FC0), "rows left unwritten"
        ok, ratio, frob = OQ.check_bf16_result(got, R, S)
        assert ok, (ratio, frob)


@pytest.mark.parametrize("bits", [4, 3, 1])
def test_grouped_decode_bias_scale2_ragged(bits):
    """Grouped calls of a few rows per expert (the grouped decode kernel): ragged N, tiles
    shorter than 8 rows, a bias per expert and second-level scales per expert and channel."""
    Q = qw()
    E, T, k, K, N = 16, 6, 4, 1024, 264
    p = synth.w4a16_problem(T, N, K, bits=bits, E=E, cfg_id=1200 + bits, bias=True)
    logits = synth.router_logits(T, E, cfg_id=1201)
    wfmt = {4: Q.QW_W_INT4_G128_BF16, 3: Q.QW_W_INT3_G128_BF16,
            1: Q.QW_W_INT1_G128_BF16}[bits] | Q.QW_W_SCALE2
    d, wp, sp_ = repack(wfmt, E, N, K, p["w_canon"], p["s_canon"])
    rng = np.random.default_rng(1202)
    t = (2.0 ** rng.integers(-2, 3, (E, N))).astype(np.float32)
    err = Q.new_error_flag()
    Q.qw_repack_scale2(d, dev(t), sp_, err)
    ids, spairs, off = route(logits, k)
    P = T * k
    A = dev(p["A"].view(np.int16))
    As = torch.empty((P, K), dtype=torch.int16, device="cuda")
    sp_dev, off_dev = dev(spairs.astype(np.int32)), dev(off.astype(np.int32))
    Q.qgemm_moe_permute(Q.QW_A_BF16, A, None, K, sp_dev, P, k, As, None)
    C = torch.full((P, N), -1, dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_BF16, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    Q.qgemm_moe_grouped(d, wp, sp_, Q.QW_A_BF16, As, None, off_dev, P,
                        dev(p["bias"].view(np.int16)), C, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    tok = spairs // k
    e_of = np.searchsorted(off, np.arange(P), side="right") - 1
    Cn = u16_view(C)
    Rall, Sall = np.zeros((P, N)), np.zeros((P, N))
    for e in np.unique(e_of):
        sel = np.nonzero(e_of == e)[0]
        R, S = OQ.w4a16_from_canonical(p["A"][tok[sel]], p["w_canon"][e], p["s_canon"][e], K,
                                       bits)
        Rall[sel], Sall[sel] = OQ.apply_scale2(R, S, t[e], p["bias"][e])
    ok, ratio, frob = OQ.check_bf16_result(Cn, Rall, Sall)
    assert ok, (ratio, frob)


@pytest.mark.parametrize("T", [80, 160, 240])
@pytest.mark.parametrize("bits", [4, 3, 2, 1])
def test_grouped_wide_token_tiles_bias_scale2_ragged(T, bits):
    """Grouped calls of 10 to 30 rows per expert on average (E=16, top-2): T=80 runs the
    grouped GEMV (16-row tiles), T=160 and 240 the tcgen05 path with partly filled 128-token
    tiles.  Expert 0 takes every token (its logit is raised), so it spans several tiles;
    ragged N, K of ten groups (a partial second stage), a bias per expert and second-level
    scales."""
    Q = qw()
    E, k, K, N = 16, 2, 1280, 264
    p = synth.w4a16_problem(T, N, K, bits=bits, E=E, cfg_id=1300 + bits, bias=True)
    logits = synth.router_logits(T, E, cfg_id=1301 + T)
    logits[:, 0] += 100.0
    wfmt = {4: Q.QW_W_INT4_G128_BF16, 3: Q.QW_W_INT3_G128_BF16, 2: Q.QW_W_INT2_G128_BF16,
            1: Q.QW_W_INT1_G128_BF16}[bits] | Q.QW_W_SCALE2
    d, wp, sp_ = repack(wfmt, E, N, K, p["w_canon"], p["s_canon"])
    rng = np.random.default_rng(1302)
    t = (2.0 ** rng.integers(-2, 3, (E, N))).astype(np.float32)
    err = Q.new_error_flag()
    Q.qw_repack_scale2(d, dev(t), sp_, err)
    ids, spairs, off = route(logits, k)
    P = T * k
    assert off[1] - off[0] == T
    A = dev(p["A"].view(np.int16))
    As = torch.empty((P, K), dtype=torch.int16, device="cuda")
    sp_dev, off_dev = dev(spairs.astype(np.int32)), dev(off.astype(np.int32))
    Q.qgemm_moe_permute(Q.QW_A_BF16, A, None, K, sp_dev, P, k, As, None)
    C = torch.full((P, N), -1, dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_BF16, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    Q.qgemm_moe_grouped(d, wp, sp_, Q.QW_A_BF16, As, None, off_dev, P,
                        dev(p["bias"].view(np.int16)), C, ws, wsn, err)
    assert Q.qw_read_error(err) == 0
    tok = spairs // k
    e_of = np.searchsorted(off, np.arange(P), side="right") - 1
    Cn = u16_view(C)
    Rall, Sall = np.zeros((P, N)), np.zeros((P, N))
    for e in np.unique(e_of):
        sel = np.nonzero(e_of == e)[0]
        R, S = OQ.w4a16_from_canonical(p["A"][tok[sel]], p["w_canon"][e], p["s_canon"][e], K,
                                       bits)
        Rall[sel], Sall[sel] = OQ.apply_scale2(R, S, t[e], p["bias"][e])
    ok, ratio, frob = OQ.check_bf16_result(Cn, Rall, Sall)
    assert ok, (ratio, frob)
