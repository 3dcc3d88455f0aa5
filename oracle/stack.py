"""The fp64 oracle: plain definitions, one sequence at a time.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every function cites
the passage it restates.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from typing import Optional, Sequence

import numpy as np
from scipy.special import erf as _erf

ABS_TOL = 2e-3   # absolute rail of the graded rule
REL_TOL = 2e-2   # relative rail of the graded rule


def layer_norm(z: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float = 1e-5) -> np.ndarray:
    """Row LayerNorm over the last axis: (z - mean) / sqrt(var + eps) * gamma + beta.

    Mean and biased variance (divide by D) over the D columns of each row;
    eps inside the square root.  The pages keep these statistics in fp32 and
    compute the variance in two passes ("TikTok TechJam 2026 -- Problem 3",
    section 3, one-pass variance rejected); here they are exact in float64.
    """
    z = np.asarray(z, dtype=np.float64)
    mu = z.mean(axis=-1, keepdims=True)
    var = ((z - mu) ** 2).mean(axis=-1, keepdims=True)
    return (z - mu) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def gelu(z: np.ndarray) -> np.ndarray:
    """Exact GELU, 0.5 z (1 + erf(z / sqrt 2)).

    "TikTok TechJam 2026 -- Problem 3", section 2.3: the scored path uses the
    exact erf GELU (the cuBLASLt tanh epilogue was only a candidate).
    """
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1.0 + _erf(z / np.sqrt(2.0)))


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_heads: int,
              length: int, causal: bool, q_pos: Optional[np.ndarray] = None,
              return_probs: bool = False):
    """Multi-head scaled-dot-product attention of one sequence, textbook form.

    "TikTok TechJam 2026 -- Problem 3", section 2.1, steps (1)-(5):
    S = Q K^T, S / sqrt(d_k), mask, row softmax over keys, A V.  Head h owns
    columns [h*hd, (h+1)*hd) of q, k and v (the fused QKV output viewed per
    head, section 2.2).

    q: [nq, D] queries at positions ``q_pos`` (default 0..nq-1);
    k, v: [nk, D] keys/values at positions 0..nk-1.
    Allowed (query i, key j): j < length (right-padded key mask, section 2.1
    "the mask trick"), and j <= pos(i) when causal.
    A query with no allowed key gets a zero output.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    nq, D = q.shape
    nk = k.shape[0]
    hd = D // n_heads
    if q_pos is None:
        q_pos = np.arange(nq)
    j = np.arange(nk)
    allowed = (j[None, :] < length)
    if causal:
        allowed = allowed & (j[None, :] <= np.asarray(q_pos)[:, None])
    any_allowed = allowed.any(axis=1)
    out = np.zeros((nq, D), dtype=np.float64)
    probs = [] if return_probs else None
    for h in range(n_heads):
        cols = slice(h * hd, (h + 1) * hd)
        s = q[:, cols] @ k[:, cols].T                      # (1) scores
        s = s / np.sqrt(hd)                                 # (2) scale
        s = np.where(allowed, s, -np.inf)                   # (3) mask
        m = np.max(s, axis=1, keepdims=True)                # (4) softmax over keys
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.where(allowed, np.exp(s - m), 0.0)
        den = e.sum(axis=1, keepdims=True)
        p = np.where(any_allowed[:, None], e / np.where(den > 0, den, 1.0), 0.0)
        out[:, cols] = p @ v[:, cols]                       # (5) weighted values
        if return_probs:
            probs.append(p)
    if return_probs:
        return out, np.stack(probs)
    return out


def sequence_forward(params, n_heads: int, xs: np.ndarray, length: int, causal: bool,
                     norm_placement: int = 0, eps: float = 1e-5,
                     q_rows: Optional[np.ndarray] = None) -> np.ndarray:
    """The L-layer stack on one sequence; returns fp64 output rows.

    Per layer ("TikTok TechJam 2026 -- Problem 3", section 1.A and 2.2):
      a  = LN1(h)                    (pre-LN; post-LN reads h itself)
      q, k, v = a Wq^T + bq, a Wk^T + bk, a Wv^T + bv   (fused QKV)
      h  = h + attention(q, k, v) Wo^T + bo              (o_proj + residual)
      a2 = LN2(h)
      h  = h + GELU(a2 W1^T + b1) W2^T + b2              (FFN + residual)
    Post-LN (norm_placement=1): h = LN1(h + attn(h)), h = LN2(h + FFN(h)).
    Tail: y = LN_f(h), rows at positions >= length set to zero.

    ``xs`` holds positions 0..len(xs)-1.  With ``q_rows`` given, the last
    layer is evaluated only at those positions (earlier layers at every row
    of ``xs``), which is exact when ``xs`` covers every key those rows may
    attend to.
    """
    h = np.asarray(xs, dtype=np.float64)
    L = len(params.layers)
    H = int(n_heads)
    for l, P in enumerate(params.layers):
        last = (l == L - 1)
        rows = q_rows if (last and q_rows is not None) else None
        a = layer_norm(h, P.ln1_g, P.ln1_b, eps) if norm_placement == 0 else h
        aq = a if rows is None else a[rows]
        q = aq @ P.wq.astype(np.float64).T + P.bq
        k = a @ P.wk.astype(np.float64).T + P.bk
        v = a @ P.wv.astype(np.float64).T + P.bv
        o = attention(q, k, v, H, length, causal, q_pos=None if rows is None else rows)
        hr = h if rows is None else h[rows]
        t = hr + o @ P.wo.astype(np.float64).T + P.bo
        if norm_placement == 1:
            t = layer_norm(t, P.ln1_g, P.ln1_b, eps)
            a2 = t
        else:
            a2 = layer_norm(t, P.ln2_g, P.ln2_b, eps)
        f = gelu(a2 @ P.w1.astype(np.float64).T + P.b1) @ P.w2.astype(np.float64).T + P.b2
        h = t + f
        if norm_placement == 1:
            h = layer_norm(h, P.ln2_g, P.ln2_b, eps)
    y = layer_norm(h, params.lnf_g, params.lnf_b, eps)
    pos = np.arange(y.shape[0]) if q_rows is None else np.asarray(q_rows)
    y[pos >= length] = 0.0
    return y


def forward(params, n_heads: int, x: np.ndarray, lengths: Optional[np.ndarray], causal: bool,
            norm_placement: int = 0, eps: float = 1e-5,
            batches: Optional[Sequence[int]] = None,
            rows: Optional[np.ndarray] = None, threads: int = 0) -> np.ndarray:
    """The whole forward, sequence by sequence (sequences are independent).

    x: float32 [nb, S, D] holding the sequences listed in ``batches`` (all of
    them when ``batches`` is None); lengths: int [B] for the full batch or
    None (every sequence full).  With ``rows`` given (sorted positions), only
    those output rows are computed for each sequence, from the causal prefix
    when ``causal`` (exact), else from the whole sequence.
    Returns float64 [nb, S or len(rows), D].
    """
    x = np.asarray(x)
    nb, S, D = x.shape
    if batches is None:
        batches = list(range(nb))
    if lengths is None:
        lens = [S] * nb
    else:
        lens = [int(lengths[b]) for b in batches]

    def one(i):
        if rows is None:
            return sequence_forward(params, n_heads, x[i], lens[i], causal, norm_placement, eps)
        r = np.asarray(rows)
        prefix = int(r.max()) + 1 if causal else S
        return sequence_forward(params, n_heads, x[i, :prefix], lens[i], causal, norm_placement, eps, q_rows=r)

    nthr = threads or min(nb, max(1, (os.cpu_count() or 1) // 2))
    if nthr <= 1 or nb == 1:
        outs = [one(i) for i in range(nb)]
    else:
        with _cf.ThreadPoolExecutor(nthr) as ex:
            outs = list(ex.map(one, range(nb)))
    return np.stack(outs)


def attention_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray, n_heads: int,
                       length: int, causal: bool, return_intermediates: bool = False):
    """Gradients (dq, dk, dv) of the attention of ``attention`` for one sequence.

    The gradient of O = softmax(Q K^T / sqrt(d_k) + mask) V ("TikTok TechJam 2026 --
    Problem 3", section 2.1) by the chain rule, per head:
      dV = P^T dO;  dP = dO V^T;  dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik);
      dQ = dS K / sqrt(d_k);  dK = dS^T Q / sqrt(d_k).
    sum_k P_ik dP_ik equals dO_i . O_i, the row sum the fused backward of
    "Training throughput baseline" (Fused attention) takes from the output gradient
    and the output.  Query rows at or past ``length`` are padding: their output
    gradient is ignored (taken as zero), so their dq is zero and they add nothing
    to dk and dv; keys at or past ``length`` are masked and get zero gradient.
    q, k, v, dout: [S, D].  Returns float64 dq, dk, dv [S, D] (and, with
    ``return_intermediates``, the per-head P and dS, [H, S, S] each).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.array(dout, dtype=np.float64)
    S, D = q.shape
    hd = D // n_heads
    do[length:] = 0.0
    j = np.arange(S)
    allowed = (j[None, :] < length)
    if causal:
        allowed = allowed & (j[None, :] <= j[:, None])
    any_allowed = allowed.any(axis=1, keepdims=True)
    dq = np.zeros((S, D))
    dk = np.zeros((S, D))
    dv = np.zeros((S, D))
    ps, dss = [], []
    for h in range(n_heads):
        c = slice(h * hd, (h + 1) * hd)
        s = np.where(allowed, q[:, c] @ k[:, c].T / np.sqrt(hd), -np.inf)
        m = np.max(s, axis=1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.where(allowed, np.exp(s - m), 0.0)
        den = e.sum(axis=1, keepdims=True)
        p = np.where(any_allowed, e / np.where(den > 0, den, 1.0), 0.0)
        dv[:, c] = p.T @ do[:, c]
        dp = do[:, c] @ v[:, c].T
        ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
        dq[:, c] = ds @ k[:, c] / np.sqrt(hd)
        dk[:, c] = ds.T @ q[:, c] / np.sqrt(hd)
        if return_intermediates:
            ps.append(p)
            dss.append(ds)
    if return_intermediates:
        return dq, dk, dv, np.stack(ps), np.stack(dss)
    return dq, dk, dv


def attention_lse(q: np.ndarray, k: np.ndarray, n_heads: int, length: int, causal: bool) -> np.ndarray:
    """Natural log of the softmax normaliser of every (head, query row) of ``attention``:
    LSE_hi = log sum_{allowed j} exp(q_i . k_j / sqrt(d_k)); -inf where no key is allowed.
    Returns float64 [n_heads, S]."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    S, D = q.shape
    hd = D // n_heads
    j = np.arange(S)
    allowed = (j[None, :] < length)
    if causal:
        allowed = allowed & (j[None, :] <= j[:, None])
    out = np.full((n_heads, S), -np.inf)
    for h in range(n_heads):
        c = slice(h * hd, (h + 1) * hd)
        s = np.where(allowed, q[:, c] @ k[:, c].T / np.sqrt(hd), -np.inf)
        m = np.max(s, axis=1)
        ok = np.isfinite(m)
        mm = np.where(ok, m, 0.0)
        tot = np.where(allowed, np.exp(s - mm[:, None]), 0.0).sum(axis=1)
        out[h] = np.where(ok, mm + np.log(np.where(ok, tot, 1.0)), -np.inf)
    return out


def attention_batched(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_heads: int,
                      lengths: np.ndarray, causal: bool) -> np.ndarray:
    """``attention`` for a batch of sequences at once: q, k, v [nb, S, D], lengths [nb].

    The same five steps of "TikTok TechJam 2026 -- Problem 3", section 2.1
    (scores, 1/sqrt(d_k) scale, mask, row softmax over keys, weighted values),
    applied to every sequence and head together; sequence b allows key j for
    query i iff j < lengths[b] (and j <= i when causal).  A query with no
    allowed key gets a zero output.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    nb, S, D = q.shape
    hd = D // n_heads
    j = np.arange(S)
    allowed = np.broadcast_to((j[None, :] < np.asarray(lengths)[:, None])[:, None, :], (nb, S, S))
    if causal:
        allowed = allowed & (j[None, :] <= j[:, None])[None]
    allowed = allowed[:, None]                                          # [nb, 1, S, S]
    any_allowed = allowed.any(axis=-1, keepdims=True)
    heads = lambda t: t.reshape(nb, S, n_heads, hd).transpose(0, 2, 1, 3)  # [nb, H, S, hd]
    qh, kh, vh = heads(q), heads(k), heads(v)
    s = qh @ kh.transpose(0, 1, 3, 2)                                   # (1) scores
    s = s / np.sqrt(hd)                                                 # (2) scale
    s = np.where(allowed, s, -np.inf)                                   # (3) mask
    m = np.max(s, axis=-1, keepdims=True)                               # (4) softmax over keys
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.where(allowed, np.exp(s - m), 0.0)
    den = e.sum(axis=-1, keepdims=True)
    p = np.where(any_allowed, e / np.where(den > 0, den, 1.0), 0.0)
    o = p @ vh                                                          # (5) weighted values
    return o.transpose(0, 2, 1, 3).reshape(nb, S, D)


def _chunk_forward(params, n_heads: int, xs: np.ndarray, lens: np.ndarray, causal: bool,
                   norm_placement: int, eps: float) -> np.ndarray:
    """``sequence_forward`` for a chunk of sequences [nb, S, D] with lengths [nb]."""
    nb, S, D = xs.shape
    # tokens of all sequences as the rows of one matrix for the linear layers
    h = np.asarray(xs, dtype=np.float64).reshape(nb * S, D)
    seq = lambda t: t.reshape(nb, S, -1)
    for P in params.layers:
        a = layer_norm(h, P.ln1_g, P.ln1_b, eps) if norm_placement == 0 else h
        q = a @ P.wq.astype(np.float64).T + P.bq
        k = a @ P.wk.astype(np.float64).T + P.bk
        v = a @ P.wv.astype(np.float64).T + P.bv
        o = attention_batched(seq(q), seq(k), seq(v), n_heads, lens, causal).reshape(nb * S, D)
        t = h + o @ P.wo.astype(np.float64).T + P.bo
        if norm_placement == 1:
            t = layer_norm(t, P.ln1_g, P.ln1_b, eps)
            a2 = t
        else:
            a2 = layer_norm(t, P.ln2_g, P.ln2_b, eps)
        f = gelu(a2 @ P.w1.astype(np.float64).T + P.b1) @ P.w2.astype(np.float64).T + P.b2
        h = t + f
        if norm_placement == 1:
            h = layer_norm(h, P.ln2_g, P.ln2_b, eps)
    y = seq(layer_norm(h, params.lnf_g, params.lnf_b, eps))
    y[np.arange(S)[None, :] >= np.asarray(lens)[:, None]] = 0.0
    return y


def _chunk_task(args):
    return _chunk_forward(*args)


_POOL = None


def _process_pool():
    """A pool of one worker process per core, started with ``spawn`` and kept for
    the life of the process.  Each worker runs single-threaded BLAS: many small
    array operations in parallel processes beat threads that contend for one
    multi-threaded BLAS."""
    global _POOL
    if _POOL is None:
        import atexit
        import multiprocessing as mp
        keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
        saved = {k: os.environ.get(k) for k in keys}
        for k in keys:
            os.environ[k] = "1"
        try:
            _POOL = mp.get_context("spawn").Pool(max(1, os.cpu_count() or 1))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        atexit.register(_POOL.terminate)
    return _POOL


def forward_batched(params, n_heads: int, x: np.ndarray, lengths: Optional[np.ndarray], causal: bool,
                    norm_placement: int = 0, eps: float = 1e-5, chunk: int = 0,
                    processes: bool = False) -> np.ndarray:
    """The whole forward of ``forward`` (same layer order, masks and tail), with the
    sequences taken ``chunk`` at a time through batched array operations instead of
    one at a time.  Sequences are independent, so this is the same definition
    evaluated for many sequences per array operation.

    With ``processes`` the chunks are spread over a pool of worker processes
    (see ``_process_pool``); otherwise they run one after another in this process.

    x: float32 [nb, S, D]; lengths: int [nb] or None.  Returns float64 [nb, S, D].
    """
    x = np.asarray(x)
    nb, S, D = x.shape
    lens = np.full(nb, S, dtype=np.int64) if lengths is None else np.asarray(lengths, dtype=np.int64)
    if chunk <= 0:
        # about 64 MB of fp64 scores per chunk
        chunk = max(1, min(nb, (64 << 20) // (8 * n_heads * S * S)))
    starts = list(range(0, nb, chunk))
    tasks = [(params, n_heads, x[s0:s0 + chunk], lens[s0:s0 + chunk], causal, norm_placement, eps)
             for s0 in starts]
    if processes and len(tasks) > 1:
        parts = _process_pool().map(_chunk_task, tasks)
    else:
        parts = [_chunk_task(t) for t in tasks]
    return np.concatenate(parts, axis=0)


def gate(u: np.ndarray, r: np.ndarray) -> np.ndarray:
    """Elementwise acceptance: |u - r| <= 2e-3 or |u - r| <= 0.02 |r|.

    The graded rule stated on "Transformerkernel" (Inspiration) and on
    "Shape-specialized Transformer Inference on Commodity GPUs" (How this
    solution addresses the problem statement), and the 2e-3 absolute budget
    of "TikTok TechJam 2026 -- Problem 3", section 2.3.
    """
    u = np.asarray(u, np.float64)
    r = np.asarray(r, np.float64)
    d = np.abs(u - r)
    return (d <= ABS_TOL) | (d <= REL_TOL * np.abs(r))
