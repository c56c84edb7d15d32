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
    wfmt = {4: Q.QW_W_INT4_G128_BF16, 3: Q.QW_W_INT3_G128_BF16,
            2: Q.QW_W_INT2_G128_BF16}[prob["bits"]]
    d, wp, sp = repack(wfmt, 1, prob["N"], prob["K"], prob["w_canon"], prob["s_canon"])
    A = dev(prob["A"].view(np.int16))
    M = prob["A"].shape[0] if M is None else M
    C = torch.full((M, prob["N"]), -1, dtype=torch.int16, device="cuda")
    b = None if bias is None else dev(bias.view(np.int16))
    ws_n = Q.qgemm_workspace_size(d, Q.QW_A_BF16, M)
    ws = torch.zeros(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_dense(d, wp, sp, Q.QW_A_BF16, A, None, b, C, M, ws, ws_n, err)
    assert Q.qw_read_error(err) == 0
    return u16_view(C)


def dense_fp8w(prob, bias=None):
    """FP8-weight WnA16 (E4M3 codes, BF16 group-128 scales) through qgemm_dense."""
    Q = qw()
    N, K = prob["N"], prob["K"]
    d, wp, sp = repack(Q.QW_W_FP8E4M3_G128_BF16, 1, N, K, prob["w_canon"], prob["s_canon"])
    M = prob["A"].shape[0]
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    b = None if bias is None else dev(bias.view(np.int16))
    wsn = Q.qgemm_workspace_size(d, Q.QW_A_BF16, M)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")
    err = Q.new_error_flag()
    Q.qgemm_dense(d, wp, sp, Q.QW_A_BF16, dev(prob["A"].view(np.int16)), None, b, C, M, ws, wsn,
                  err)
    assert Q.qw_read_error(err) == 0
    return u16_view(C)


def dense_w4a8(prob, bias=None, wfmt=None, workspace=True):
    Q = qw()
    wfmt = Q.QW_W_MXFP4_G32 if wfmt is None else wfmt
    d, wp, sp = repack(wfmt, 1, prob["N"], prob["K"], prob["w_canon"], prob["s_canon"])
    A = dev(prob["A"])
    Asf = dev(prob["A_sf"])
    M = prob["A"].shape[0]
    C = torch.full((M, prob["N"]), -1, dtype=torch.int16, device="cuda")
    b = None if bias is None else dev(bias.view(np.int16))
    # the workspace the call asks for (none for a dense call today)
    ws_n = Q.qgemm_workspace_size(d, Q.QW_A_MXFP8_G32, M) if workspace else 0
    ws = torch.zeros(max(ws_n, 16), dtype=torch.uint8, device="cuda") if workspace else None
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


# ----------------------------------------------------------------------------- full-size MoE
def moe_pipeline(afmt, wfmt, E, T, K, N, topk, cfg_id, bits=4, weights=None, x_sorted=None,
                 route_from=None, replicas=1):
    """Route -> permute -> grouped GEMM through the C ABI on device-generated inputs.
    Returns a dict of device tensors (inputs and outputs) for sampled oracle checks.
    ``route_from`` reuses another pipeline's routing (e.g. the down projection after the
    up projection); its ``route`` step then does nothing.  ``replicas`` > 1 keeps that many
    copies of the packed weights; ``gemm(i)`` reads copy i mod replicas (timing loops use
    it so that consecutive steps do not find the weights in L2)."""
    import synth
    import synth.device as sd
    Q = qw()
    P = T * topk
    logits = synth.router_logits(T, E, cfg_id=cfg_id)
    lg = dev(logits)
    if weights is None:
        weights = (sd.mxfp4_weights(E, N, K, cfg_id=cfg_id) if wfmt == Q.QW_W_MXFP4_G32
                   else sd.int_weights(E, N, K, bits=bits, cfg_id=cfg_id))
    w_canon, s_canon = weights
    d = Q.qw_repack_query(wfmt, E, N, K)
    wp, spk = Q.empty_packed(d)
    err = Q.new_error_flag()
    Q.qw_repack(d, w_canon, s_canon, wp, spk, err)
    assert Q.qw_read_error(err) == 0
    ids = torch.empty((max(T, 1), topk), dtype=torch.int32, device="cuda")
    sp = torch.empty((max(P, 1),), dtype=torch.int32, device="cuda")
    off = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
    n = Q.qgemm_moe_route_workspace_size(T, E, topk)
    rws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    out = dict(logits=logits, logits_dev=lg, w_canon=w_canon, s_canon=s_canon, desc=d, wp=wp,
               sp_packed=spk, sorted_pairs=sp, offsets=off, topk_ids=ids)

    def route(i=0):
        Q.qgemm_moe_route(lg, T, E, topk, ids, sp, off, rws, n)

    if route_from is not None:
        ids, sp, off = route_from["topk_ids"], route_from["sorted_pairs"], route_from["offsets"]
        out.update(sorted_pairs=sp, offsets=off, topk_ids=ids, logits=route_from["logits"])

        def route(i=0):  # noqa: F811  (routing shared with `route_from`)
            pass

    if afmt == Q.QW_A_MXFP8_G32:
        A, Asf = sd.mxfp8_activations(T, K, cfg_id=cfg_id)
        As = torch.empty((P, K), dtype=torch.uint8, device="cuda")
        Asf_s = torch.empty((P, K // 32), dtype=torch.uint8, device="cuda")
        out.update(A=A, A_sf=Asf)
    else:
        A = sd.bf16_activations(T, K, cfg_id=cfg_id) if x_sorted is None else None
        As = torch.empty((P, K), dtype=torch.int16, device="cuda") if x_sorted is None else x_sorted
        Asf, Asf_s = None, None
        out.update(A=A)

    def permute(i=0):
        if x_sorted is None:
            Q.qgemm_moe_permute(afmt, A, Asf, K, sp, P, topk, As, Asf_s)

    C = torch.empty((P, N), dtype=torch.int16, device="cuda")
    wsn = Q.qgemm_workspace_size(d, afmt, P)
    ws = torch.zeros(max(wsn, 16), dtype=torch.uint8, device="cuda")

    wps = [(wp, spk)] + [(wp.clone(), spk.clone()) for _ in range(replicas - 1)]

    def set_replicas(r):
        """Keep r copies of the packed weights (r >= 1)."""
        del wps[max(1, r):]
        wps.extend((wp.clone(), spk.clone()) for _ in range(r - len(wps)))

    def gemm(i=0):
        w, s = wps[i % len(wps)]
        Q.qgemm_moe_grouped(d, w, s, afmt, As, Asf_s, off, P, None, C, ws, wsn, err)

    def gemm_indexed(i=0):
        """The Indexed path: the grouped GEMM reading the unpermuted activations by pair id
        (MX formats; replaces permute + gemm)."""
        w, s = wps[i % len(wps)]
        Q.qgemm_moe_grouped_indexed(d, w, s, afmt, A, Asf, T, sp, topk, off, P, None, C, ws,
                                    wsn, err)

    out.update(A_sorted=As, A_sf_sorted=Asf_s, C=C, err=err, route=route, permute=permute,
               gemm=gemm, gemm_indexed=gemm_indexed, set_replicas=set_replicas)
    return out


def sample_rows_per_expert(offsets, per_expert=2, max_experts=None, seed=0):
    """Row indices of the grouped output: the first, last (and a middle) row of sampled
    non-empty experts, always including the largest and smallest non-empty ones."""
    off = np.asarray(offsets, dtype=np.int64)
    counts = np.diff(off)
    nz = np.nonzero(counts)[0]
    if max_experts is not None and nz.size > max_experts:
        rng = np.random.default_rng(seed)
        keep = set(rng.choice(nz, max_experts - 2, replace=False).tolist())
        keep |= {int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])}
        nz = np.array(sorted(keep))
    rows = []
    for e in nz:
        b, c = off[e], counts[e]
        cand = [b, b + c - 1, b + c // 2][:max(1, per_expert)]
        rows.extend(sorted(set(int(r) for r in cand)))
    return np.array(rows, dtype=np.int64)
