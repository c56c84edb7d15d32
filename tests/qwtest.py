"""Test helpers: move synthetic problems to the GPU and run them through the C ABI.

No arithmetic of the method here - only buffer handling around the library calls.
"""
import numpy as np
import torch


def qw():
    import moe_qw_repack_gb300.qw as q
    return q


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def u16_view(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def repack(wfmt, E, N, K, w_canon, s_canon):
    """Repack canonical weights (numpy or device tensors) -> (desc, w_packed, s_packed)."""
    Q = qw()
    d = Q.qw_repack_query(wfmt, E, N, K)
    wc = w_canon if isinstance(w_canon, torch.Tensor) else dev(w_canon)
    sc = s_canon if isinstance(s_canon, torch.Tensor) else dev(s_canon)
    wp, sp = Q.empty_packed(d)
    err = Q.new_error_flag()
    Q.qw_repack(d, wc, sc, wp, sp, err)
    code = Q.qw_read_error(err)
    assert code == 0, f"repack error flag {code}"
    return d, wp, sp


def dense_w4a16(prob, bias=None, M=None):
    Q = qw()
    wfmt = Q.QW_W_INT4_G128_BF16 if prob["bits"] == 4 else Q.QW_W_INT3_G128_BF16
    d, wp, sp = repack(wfmt, 1, prob["N"], prob["K"], prob["w_canon"], prob["s_canon"])
    A = dev(prob["A"].view(np.int16))
    M = prob["A"].shape[0] if M is None else M
    C = torch.full((M, prob["N"]), -1, dtype=torch.int16, device="cuda")
    b = None if bias is None else dev(bias.view(np.int16))
    ws_n = Q.qgemm_workspace_size(d, Q.QW_A_BF16, M)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_dense(d, wp, sp, Q.QW_A_BF16, A, None, b, C, M, ws, ws_n, err)
    assert Q.qw_read_error(err) == 0
    return u16_view(C)


def dense_w4a8(prob, bias=None):
    Q = qw()
    d, wp, sp = repack(Q.QW_W_MXFP4_G32, 1, prob["N"], prob["K"], prob["w_canon"],
                       prob["s_canon"])
    A = dev(prob["A"])
    Asf = dev(prob["A_sf"])
    M = prob["A"].shape[0]
    C = torch.full((M, prob["N"]), -1, dtype=torch.int16, device="cuda")
    b = None if bias is None else dev(bias.view(np.int16))
    ws_n = Q.qgemm_workspace_size(d, Q.QW_A_MXFP8_G32, M)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_dense(d, wp, sp, Q.QW_A_MXFP8_G32, A, Asf, b, C, M, ws, ws_n, err)
    code = Q.qw_read_error(err)
    assert code == 0, f"error flag {code}"
    return u16_view(C)


def route(logits_np, topk):
    Q = qw()
    T, E = logits_np.shape
    lg = dev(logits_np)
    ids = torch.full((max(T, 1), topk), -1, dtype=torch.int32, device="cuda")
    sp = torch.full((max(T * topk, 1),), -1, dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    n = Q.qgemm_moe_route_workspace_size(T, E, topk)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_moe_route(lg, T, E, topk, ids, sp, off, ws, n, err)
    assert Q.qw_read_error(err) == 0
    return host(ids)[:T], host(sp)[:T * topk], host(off)
