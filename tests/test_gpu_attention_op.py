"""Attention on its own: forward with the row log-sum-exp, and the backward (dq, dk, dv).

"Training throughput baseline" (Fused attention) keeps the log-sum-exp in the
forward and rebuilds the probabilities from it in a backward split into a
query-tile kernel (dQ) and a key-tile kernel (dK, dV).  Inputs are fp16 (q, k, v,
dO) and the oracle runs in fp64 on the same values.  The kernels round P and dS
to fp16 once (unit roundoff u = 2^-11) and accumulate in fp32, and the row sums D
come from the fp16 output, so each element is held to the first-order bound of
those roundings, doubled (the oracle's own P and dS give the bound):
  o     2u (sum_j P|v_j| + |o|)
  dv    2u' sum_i P_ij |dO_i|
  dq    2 sum_j (u'|dS_ij| + P_ij dD_i) |k_j| / sqrt(hd)
  dk    2 sum_i (u'|dS_ij| + P_ij dD_i) |q_i| / sqrt(hd)
with u' = u + 1e-5 (fp32 score and exponential error) and dD_i = sum_d |dO_id| x
the bound on o_id; plus 1e-6 absolute.  lse must match to 1e-4 (log2 units).
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

U = 2.0 ** -11
U1 = U + 1e-5
LOG2E = 1.4426950408889634


def _run(B, S, H, hd, causal, lens, seed):
    import torch
    import attention_qkv_gemm_gb300 as pkg
    rng = np.random.default_rng(seed)
    D = H * hd
    qkv = rng.standard_normal((B, S, 3 * D)).astype(np.float16)
    dout = rng.standard_normal((B, S, D)).astype(np.float16)
    a = pkg.tfl_attn_create(B, S, H, hd)
    try:
        st = torch.cuda.current_stream().cuda_stream
        qd = torch.from_numpy(qkv).cuda()
        dod = torch.from_numpy(dout).cuda()
        ld = None if lens is None else torch.from_numpy(np.asarray(lens, np.int32)).cuda()
        o = torch.full((B, S, D), float("nan"), dtype=torch.float16, device="cuda")
        lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device="cuda")
        dqkv = torch.full((B, S, 3 * D), float("nan"), dtype=torch.float32, device="cuda")
        lp = None if ld is None else ld.data_ptr()
        pkg.tfl_attn_forward(a, qd.data_ptr(), lp, int(causal), o.data_ptr(), lse.data_ptr(), st)
        pkg.tfl_attn_backward(a, qd.data_ptr(), o.data_ptr(), dod.data_ptr(), lse.data_ptr(), lp, int(causal),
                              dqkv.data_ptr(), st)
        assert pkg.tfl_attn_status(a, st) == 0, pkg.tfl_last_error()
        return qkv, dout, o.cpu().numpy(), lse.cpu().numpy(), dqkv.cpu().numpy()
    finally:
        pkg.tfl_attn_destroy(a)


def _check(u, r, bound, what):
    if u.size == 0:
        return 0.0
    bad = np.abs(u - r) > bound
    assert np.isfinite(u).all(), f"{what}: non-finite"
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside the bound, "
                           f"worst |u-r|/bound {float(np.max(np.abs(u - r) / bound)):.3f}")
    return float(np.max(np.abs(u - r) / bound))


@pytest.mark.parametrize("B,S,H,hd,causal,lens", [
    (2, 300, 2, 64, True, [300, 150]),
    (2, 200, 4, 32, False, [200, 77]),
    (1, 129, 2, 64, False, None),
    (3, 64, 1, 32, True, [64, 1, 0]),
    (1, 1024, 2, 64, True, None),
    (2, 520, 3, 32, True, [519, 260]),
    # more work items than CTAs (two per SM): each CTA runs several items of 1 to 5 key
    # sub-blocks, so the forward's sub-block buffers rotate across item boundaries
    (40, 320, 8, 64, True, [320 - 7 * i for i in range(40)]),
    (64, 200, 4, 32, False, [200 - 3 * i for i in range(64)]),
])
def test_attention_forward_lse_and_backward_within_rounding_bounds(B, S, H, hd, causal, lens):
    qkv, dout, o, lse, dqkv = _run(B, S, H, hd, causal, lens, seed=S + H)
    D = H * hd
    worst = {}
    for b in range(B):
        L = S if lens is None else int(lens[b])
        q, k, v = (qkv[b, :, i * D:(i + 1) * D].astype(np.float64) for i in range(3))
        do = dout[b].astype(np.float64)
        ref_o, P = oracle.attention(q, k, v, H, L, causal, return_probs=True)
        dq, dk, dv, P2, dS = oracle.attention_backward(q, k, v, do, H, L, causal, return_intermediates=True)
        ref_lse = oracle.attention_lse(q, k, H, L, causal) * LOG2E
        for h in range(H):
            c = slice(h * hd, (h + 1) * hd)
            Ph, dSh = P2[h], dS[h]
            ob = 2 * U * (Ph @ np.abs(v[:, c]) + np.abs(ref_o[:, c])) + 1e-6
            worst["o"] = max(worst.get("o", 0), _check(o[b, :L, c].astype(np.float64), ref_o[:L, c], ob[:L],
                                                        f"o b{b} h{h}"))
            np.testing.assert_allclose(lse[b, h, :L], ref_lse[h, :L], atol=1e-4, err_msg=f"lse b{b} h{h}")
            dD = (np.abs(do[:, c]) * ob).sum(axis=1)
            dD[L:] = 0.0
            w = U1 * np.abs(dSh) + Ph * dD[:, None]
            bq = 2 * (w @ np.abs(k[:, c])) / np.sqrt(hd) + 1e-6
            bk = 2 * (w.T @ np.abs(q[:, c])) / np.sqrt(hd) + 1e-6
            dom = do.copy()
            dom[L:] = 0.0
            bv = 2 * U1 * (Ph.T @ np.abs(dom[:, c])) + 1e-6
            worst["dq"] = max(worst.get("dq", 0), _check(dqkv[b, :, c], dq[:, c], bq, f"dq b{b} h{h}"))
            worst["dk"] = max(worst.get("dk", 0), _check(dqkv[b, :, D + h * hd:D + (h + 1) * hd], dk[:, c], bk,
                                                         f"dk b{b} h{h}"))
            worst["dv"] = max(worst.get("dv", 0), _check(dqkv[b, :, 2 * D + h * hd:2 * D + (h + 1) * hd], dv[:, c],
                                                         bv, f"dv b{b} h{h}"))
        # padding rows: dq, dk, dv exactly zero
        assert np.all(dqkv[b, L:] == 0.0)
    print("\nworst |u-r|/bound:", {k_: round(v_, 3) for k_, v_ in worst.items()})
