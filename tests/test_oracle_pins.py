"""Pins of the fp64 oracle to things other than itself (CPU only).

Each oracle function is checked against a library routine (torch float64
``layer_norm``, ``gelu``, ``scaled_dot_product_attention``,
``TransformerEncoder``), a closed form, or an invariant that the definition
fixes.  ``test_planted_mistakes_are_caught`` plants plausible mistakes in the
oracle and checks that these pins catch each one.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle import stack as ofw

pytestmark = pytest.mark.filterwarnings("ignore")


def tiny_shape(B=2, S=8, D=16, H=2, F_=32, L=2, causal=True):
    return synth.Shape(B, S, D, H, F_, L, causal)


def rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# LayerNorm
# --------------------------------------------------------------------------

def test_layer_norm_matches_torch():
    r = rng(0)
    z = r.normal(size=(7, 33)) * 3 + 1
    g = r.normal(size=33)
    b = r.normal(size=33)
    ref = F.layer_norm(torch.tensor(z), (33,), torch.tensor(g), torch.tensor(b), eps=1e-5).numpy()
    np.testing.assert_allclose(oracle.layer_norm(z, g, b, 1e-5), ref, rtol=0, atol=1e-12)


def test_layer_norm_invariants():
    r = rng(1)
    z = r.normal(size=(5, 64)) * 10 - 4
    y = oracle.layer_norm(z, np.ones(64), np.zeros(64), eps=0.0)
    np.testing.assert_allclose(y.mean(-1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(-1), 1, atol=1e-12)
    beta = r.normal(size=64)
    const = np.full((3, 64), 2.5)
    np.testing.assert_allclose(oracle.layer_norm(const, r.normal(size=64), beta), np.broadcast_to(beta, (3, 64)), atol=1e-12)


# --------------------------------------------------------------------------
# GELU
# --------------------------------------------------------------------------

def test_gelu_matches_torch_and_closed_forms():
    z = np.linspace(-8, 8, 1001)
    ref = F.gelu(torch.tensor(z), approximate="none").numpy()
    np.testing.assert_allclose(oracle.gelu(z), ref, rtol=1e-14, atol=1e-15)
    # odd-part identity: gelu(z) - gelu(-z) = z
    np.testing.assert_allclose(oracle.gelu(z) - oracle.gelu(-z), z, atol=1e-14)
    assert oracle.gelu(np.array([0.0]))[0] == 0.0
    # the tanh approximation differs by > 1e-5 somewhere: the oracle is the erf form
    tanh = F.gelu(torch.tensor(z), approximate="tanh").numpy()
    assert np.max(np.abs(oracle.gelu(z) - tanh)) > 1e-5


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def _sdpa_ref(q, k, v, H, length, causal):
    nq, D = q.shape
    hd = D // H
    qt = torch.tensor(q).view(nq, H, hd).transpose(0, 1)
    kt = torch.tensor(k).view(-1, H, hd).transpose(0, 1)
    vt = torch.tensor(v).view(-1, H, hd).transpose(0, 1)
    j = torch.arange(k.shape[0])
    allowed = (j[None, :] < length).expand(nq, -1)
    if causal:
        allowed = allowed & (j[None, :] <= torch.arange(nq)[:, None])
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=allowed)
    return o.transpose(0, 1).reshape(nq, D).numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("length", [1, 5, 9])
def test_attention_matches_torch_sdpa(causal, length):
    r = rng(2)
    S, D, H = 9, 24, 3
    q, k, v = (r.normal(size=(S, D)) for _ in range(3))
    ours = oracle.attention(q, k, v, H, length, causal)
    ref = _sdpa_ref(q, k, v, H, length, causal)
    # length >= 1: key 0 is allowed for every query, so every row is defined
    np.testing.assert_allclose(ours, ref, atol=1e-12)


def test_attention_softmax_rows_sum_to_one():
    r = rng(3)
    q, k, v = (r.normal(size=(12, 16)) for _ in range(3))
    _, p = oracle.attention(q, k, v, 2, 10, True, return_probs=True)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-13)
    # no mass on padded keys or on keys after the query
    assert np.all(p[:, :, 10:] == 0)
    assert np.all(np.triu(p[0], 1) == 0)


def test_attention_single_key_equals_v():
    r = rng(4)
    q, k, v = (r.normal(size=(1, 32)) for _ in range(3))
    np.testing.assert_allclose(oracle.attention(q, k, v, 4, 1, False), v, atol=1e-14)
    # length 1 with many keys: every query sees only key 0
    q, k, v = (r.normal(size=(6, 32)) for _ in range(3))
    out = oracle.attention(q, k, v, 4, 1, False)
    np.testing.assert_allclose(out, np.broadcast_to(v[0], (6, 32)), atol=1e-14)


def test_attention_uniform_scores_average_values():
    # identical keys give equal weights: output is the mean of the allowed values
    r = rng(5)
    q = r.normal(size=(5, 8))
    k = np.tile(r.normal(size=(1, 8)), (5, 1))
    v = r.normal(size=(5, 8))
    out = oracle.attention(q, k, v, 1, 5, True)
    for i in range(5):
        np.testing.assert_allclose(out[i], v[: i + 1].mean(0), atol=1e-13)


def test_attention_scale_is_inverse_sqrt_head_dim():
    # two keys, one query: p0/p1 = exp((s0 - s1)/sqrt(hd))
    hd = 16
    q = np.zeros((1, hd)); q[0, 0] = 1.0
    k = np.zeros((2, hd)); k[0, 0] = 4.0
    v = np.zeros((2, hd)); v[0, 1] = 1.0; v[1, 2] = 1.0
    out = oracle.attention(q, k, v, 1, 2, False)
    ratio = out[0, 1] / out[0, 2]
    assert abs(ratio - np.exp(4.0 / np.sqrt(hd))) < 1e-12


# --------------------------------------------------------------------------
# Whole stack
# --------------------------------------------------------------------------

def _torch_stack(prm, shape, norm_first, eps=1e-5):
    D, H, Fd = shape.d_model, shape.n_heads, shape.d_ff
    layers = []
    for P in prm.layers:
        m = torch.nn.TransformerEncoderLayer(D, H, Fd, dropout=0.0, activation="gelu",
                                             layer_norm_eps=eps, batch_first=True,
                                             norm_first=norm_first, dtype=torch.float64)
        with torch.no_grad():
            m.self_attn.in_proj_weight.copy_(torch.tensor(np.concatenate([P.wq, P.wk, P.wv], 0)))
            m.self_attn.in_proj_bias.copy_(torch.tensor(np.concatenate([P.bq, P.bk, P.bv], 0)))
            m.self_attn.out_proj.weight.copy_(torch.tensor(P.wo))
            m.self_attn.out_proj.bias.copy_(torch.tensor(P.bo))
            m.linear1.weight.copy_(torch.tensor(P.w1)); m.linear1.bias.copy_(torch.tensor(P.b1))
            m.linear2.weight.copy_(torch.tensor(P.w2)); m.linear2.bias.copy_(torch.tensor(P.b2))
            m.norm1.weight.copy_(torch.tensor(P.ln1_g)); m.norm1.bias.copy_(torch.tensor(P.ln1_b))
            m.norm2.weight.copy_(torch.tensor(P.ln2_g)); m.norm2.bias.copy_(torch.tensor(P.ln2_b))
        m.train()  # dropout is 0; training mode keeps torch off its fused inference path
        layers.append(m)
    fn = torch.nn.LayerNorm(D, eps=eps, dtype=torch.float64)
    with torch.no_grad():
        fn.weight.copy_(torch.tensor(prm.lnf_g)); fn.bias.copy_(torch.tensor(prm.lnf_b))
    return layers, fn


def _torch_forward(prm, shape, x, lens, causal, norm_first):
    layers, fn = _torch_stack(prm, shape, norm_first)
    B, S, D = x.shape
    h = torch.tensor(x, dtype=torch.float64)
    pad = torch.arange(S)[None, :] >= torch.tensor(lens)[:, None]
    mask = torch.nn.Transformer.generate_square_subsequent_mask(S, dtype=torch.float64) if causal else None
    with torch.no_grad():
        for m in layers:
            h = m(h, src_mask=mask, src_key_padding_mask=pad, is_causal=causal)
        return fn(h).numpy()


def _batched_pool(prm, H, x, lens, causal, norm_placement=0):
    return oracle.forward_batched(prm, H, x, lens, causal, norm_placement, chunk=1, processes=True)


def _batched_inproc(prm, H, x, lens, causal, norm_placement=0):
    return oracle.forward_batched(prm, H, x, lens, causal, norm_placement, chunk=2)


@pytest.mark.parametrize("fwd", [oracle.forward, _batched_inproc, _batched_pool],
                         ids=["per_sequence", "batched", "batched_processes"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("norm_placement", [0, 1])
def test_forward_matches_torch_transformer_encoder(causal, norm_placement, fwd):
    shape = tiny_shape(B=3, S=8, D=16, H=2, F_=32, L=2, causal=causal)
    prm = synth.params(11, shape, ln_affine="random", bias_std=0.3)
    x = synth.input_x(11, shape)
    lens = np.array([8, 5, 1], dtype=np.int32)
    ours = fwd(prm, shape.n_heads, x, lens, causal, norm_placement)
    ref = _torch_forward(prm, shape, x, lens, causal, norm_first=(norm_placement == 0))
    for b in range(shape.B):
        np.testing.assert_allclose(ours[b, :lens[b]], ref[b, :lens[b]], atol=1e-11)
        assert np.all(ours[b, lens[b]:] == 0.0)


def test_zero_projections_reduce_to_final_layernorm():
    shape = tiny_shape(B=2, S=6, D=16, H=4, F_=24, L=3, causal=True)
    prm = synth.params(3, shape)
    for P in prm.layers:
        for f in synth.LayerParams.FIELDS:
            if not f.startswith("ln"):
                setattr(P, f, np.zeros_like(getattr(P, f)))
    x = synth.input_x(3, shape)
    ours = oracle.forward(prm, shape.n_heads, x, None, True)
    ref = F.layer_norm(torch.tensor(x, dtype=torch.float64), (16,), eps=1e-5).numpy()
    np.testing.assert_allclose(ours, ref, atol=1e-12)


def test_zero_output_projections_ignore_attention():
    # Wo = bo = W2 = b2 = 0: every sublayer adds zero, out = LN_f(x) whatever q/k/v are
    shape = tiny_shape(B=1, S=7, D=16, H=2, F_=32, L=2, causal=False)
    prm = synth.params(4, shape, ln_affine="random")
    for P in prm.layers:
        P.wo[:] = 0; P.bo[:] = 0; P.w2[:] = 0; P.b2[:] = 0
    x = synth.input_x(4, shape)
    ours = oracle.forward(prm, shape.n_heads, x, None, False)
    ref = F.layer_norm(torch.tensor(x, dtype=torch.float64), (16,), torch.tensor(prm.lnf_g, dtype=torch.float64),
                       torch.tensor(prm.lnf_b, dtype=torch.float64), eps=1e-5).numpy()
    np.testing.assert_allclose(ours, ref, atol=1e-12)


def test_causal_future_perturbation_leaves_prefix_unchanged():
    shape = tiny_shape(B=1, S=10, D=16, H=2, F_=32, L=2, causal=True)
    prm = synth.params(5, shape, ln_affine="random")
    x = synth.input_x(5, shape)
    base = oracle.forward(prm, 2, x, None, True)
    x2 = x.copy(); x2[0, 6:] = np.random.default_rng(1).normal(size=x2[0, 6:].shape).astype(np.float32)
    pert = oracle.forward(prm, 2, x2, None, True)
    np.testing.assert_array_equal(base[0, :6], pert[0, :6])
    assert np.max(np.abs(base[0, 6:] - pert[0, 6:])) > 1e-3


@pytest.mark.parametrize("causal", [True, False])
def test_padded_positions_have_no_effect(causal):
    shape = tiny_shape(B=1, S=10, D=16, H=2, F_=32, L=2, causal=causal)
    prm = synth.params(6, shape, ln_affine="random")
    x = synth.input_x(6, shape)
    lens = np.array([6], dtype=np.int32)
    base = oracle.forward(prm, 2, x, lens, causal)
    x2 = x.copy(); x2[0, 6:] = np.float32(100.0)
    pert = oracle.forward(prm, 2, x2, lens, causal)
    np.testing.assert_array_equal(base, pert)
    assert np.all(base[0, 6:] == 0.0)


def test_non_causal_permutation_equivariance():
    shape = tiny_shape(B=1, S=9, D=16, H=2, F_=32, L=2, causal=False)
    prm = synth.params(7, shape, ln_affine="random")
    x = synth.input_x(7, shape)
    perm = np.random.default_rng(0).permutation(9)
    a = oracle.forward(prm, 2, x, None, False)
    b = oracle.forward(prm, 2, x[:, perm], None, False)
    np.testing.assert_allclose(a[:, perm], b, atol=1e-12)


def test_seq_len_one_attention_is_value_projection():
    # one token: attention output = v = LN1(x) Wv^T + bv; whole layer by hand from library routines
    shape = tiny_shape(B=1, S=1, D=16, H=2, F_=32, L=1, causal=True)
    prm = synth.params(8, shape, ln_affine="random")
    x = synth.input_x(8, shape).astype(np.float64)[0]
    P = prm.layers[0]
    t = lambda a: torch.tensor(a, dtype=torch.float64)
    a = F.layer_norm(t(x), (16,), t(P.ln1_g), t(P.ln1_b), 1e-5)
    v = F.linear(a, t(P.wv), t(P.bv))
    h = t(x) + F.linear(v, t(P.wo), t(P.bo))
    a2 = F.layer_norm(h, (16,), t(P.ln2_g), t(P.ln2_b), 1e-5)
    h = h + F.linear(F.gelu(F.linear(a2, t(P.w1), t(P.b1))), t(P.w2), t(P.b2))
    y = F.layer_norm(h, (16,), t(prm.lnf_g), t(prm.lnf_b), 1e-5).numpy()
    ours = oracle.forward(prm, 2, synth.input_x(8, shape), None, True)[0]
    np.testing.assert_allclose(ours, y, atol=1e-12)


def test_zero_length_sequence_is_all_zero():
    shape = tiny_shape(B=2, S=5, D=16, H=2, F_=32, L=1, causal=False)
    prm = synth.params(9, shape)
    x = synth.input_x(9, shape)
    out = oracle.forward(prm, 2, x, np.array([0, 5], dtype=np.int32), False)
    assert np.all(out[0] == 0.0) and np.all(np.isfinite(out))


def test_row_sampling_matches_full_forward():
    shape = tiny_shape(B=2, S=12, D=16, H=2, F_=32, L=1, causal=True)
    prm = synth.params(10, shape, ln_affine="random")
    x = synth.input_x(10, shape)
    lens = np.array([12, 7], dtype=np.int32)
    full = oracle.forward(prm, 2, x, lens, True)
    rows = np.array([0, 3, 6, 11])
    samp = oracle.forward(prm, 2, x, lens, True, rows=rows)
    np.testing.assert_allclose(samp, full[:, rows], atol=1e-13)


def test_gate_rule():
    r = np.array([0.0, 0.0, 1.0, 1.0, -0.5, 10.0])
    u = np.array([2e-3, 2.1e-3, 1.0199, 1.0201, -0.5015, 10.19])
    assert list(oracle.gate(u, r)) == [True, False, True, False, True, True]


# --------------------------------------------------------------------------
# Planted mistakes: each must be caught by the library comparison above
# --------------------------------------------------------------------------

def _mut_scale(q, k, v, n_heads, length, causal, q_pos=None, return_probs=False):
    # scores scaled by 1/hd instead of 1/sqrt(hd)
    hd = q.shape[1] // n_heads
    return ORIG_ATTENTION(q / np.sqrt(hd), k, v, n_heads, length, causal, q_pos, return_probs)


def _mut_causal_strict(q, k, v, n_heads, length, causal, q_pos=None, return_probs=False):
    # off by one: j < i instead of j <= i (row 0 then sees nothing)
    nq = q.shape[0]
    pos = np.arange(nq) if q_pos is None else np.asarray(q_pos)
    return ORIG_ATTENTION(q, k, v, n_heads, length, causal, pos - 1 if causal else q_pos, return_probs)


def _mut_heads_transposed(q, k, v, n_heads, length, causal, q_pos=None, return_probs=False):
    # heads interleaved instead of contiguous column blocks
    nq, D = q.shape
    hd = D // n_heads
    perm = np.arange(D).reshape(hd, n_heads).T.reshape(-1)
    o = ORIG_ATTENTION(q[:, perm], k[:, perm], v[:, perm], n_heads, length, causal, q_pos, return_probs)
    inv = np.argsort(perm)
    return o[:, inv]


def _mut_unbiased_var(z, gamma, beta, eps=1e-5):
    z = np.asarray(z, np.float64)
    mu = z.mean(-1, keepdims=True)
    var = z.var(-1, ddof=1, keepdims=True)
    return (z - mu) / np.sqrt(var + eps) * gamma + beta


def _mut_tanh_gelu(z):
    return F.gelu(torch.tensor(np.asarray(z, np.float64)), approximate="tanh").numpy()


ORIG_ATTENTION = ofw.attention


@pytest.mark.parametrize("target,mut", [
    ("attention", _mut_scale),
    ("attention", _mut_causal_strict),
    ("attention", _mut_heads_transposed),
    ("layer_norm", _mut_unbiased_var),
    ("gelu", _mut_tanh_gelu),
])
def test_planted_mistakes_are_caught(monkeypatch, target, mut):
    monkeypatch.setattr(ofw, target, mut)
    shape = tiny_shape(B=2, S=8, D=16, H=2, F_=32, L=2, causal=True)
    prm = synth.params(12, shape, ln_affine="random", bias_std=0.3)
    x = synth.input_x(12, shape) * np.float32(2.0)
    lens = np.array([8, 6], dtype=np.int32)
    ours = ofw.forward(prm, 2, x, lens, True)
    ref = _torch_forward(prm, shape, x, lens, True, norm_first=True)
    diff = max(np.max(np.abs(ours[b, :lens[b]] - ref[b, :lens[b]])) for b in range(2))
    assert diff > 1e-6, f"mutation {mut.__name__} not caught (diff {diff})"


def test_dropped_bias_is_caught():
    shape = tiny_shape(B=1, S=6, D=16, H=2, F_=32, L=1, causal=True)
    prm = synth.params(13, shape, bias_std=0.3)
    x = synth.input_x(13, shape)
    ref = _torch_forward(prm, shape, x, np.array([6]), True, norm_first=True)
    # bk is left out: it adds q_i . bk to every score of row i, which softmax cancels
    for f in ("bq", "bv", "bo", "b1", "b2"):
        P = synth.params(13, shape, bias_std=0.3)
        getattr(P.layers[0], f)[:] = 0
        ours = oracle.forward(P, 2, x, None, True)
        assert np.max(np.abs(ours - ref)) > 1e-6, f


# --------------------------------------------------------------------------
# The batched attention against the library routine and planted mistakes
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_attention_batched_matches_torch_sdpa(causal):
    r = rng(21)
    nb, S, D, H = 3, 9, 24, 3
    q, k, v = (r.normal(size=(nb, S, D)) for _ in range(3))
    lens = np.array([9, 4, 1])
    ours = oracle.attention_batched(q, k, v, H, lens, causal)
    for b in range(nb):
        np.testing.assert_allclose(ours[b], _sdpa_ref(q[b], k[b], v[b], H, lens[b], causal), atol=1e-12)


def test_attention_batched_zero_length_is_zero():
    r = rng(22)
    q, k, v = (r.normal(size=(2, 5, 8)) for _ in range(3))
    out = oracle.attention_batched(q, k, v, 2, np.array([0, 5]), False)
    assert np.all(out[0] == 0.0) and np.all(np.isfinite(out))


def _bmut_scale(q, k, v, n_heads, lengths, causal):
    hd = q.shape[-1] // n_heads
    return ORIG_ATTENTION_B(q / np.sqrt(hd), k, v, n_heads, lengths, causal)


def _bmut_lengths_off_by_one(q, k, v, n_heads, lengths, causal):
    return ORIG_ATTENTION_B(q, k, v, n_heads, np.asarray(lengths) - 1, causal)


def _bmut_heads_transposed(q, k, v, n_heads, lengths, causal):
    D = q.shape[-1]
    hd = D // n_heads
    perm = np.arange(D).reshape(hd, n_heads).T.reshape(-1)
    o = ORIG_ATTENTION_B(q[..., perm], k[..., perm], v[..., perm], n_heads, lengths, causal)
    return o[..., np.argsort(perm)]


ORIG_ATTENTION_B = ofw.attention_batched


@pytest.mark.parametrize("target,mut", [
    ("attention_batched", _bmut_scale),
    ("attention_batched", _bmut_lengths_off_by_one),
    ("attention_batched", _bmut_heads_transposed),
    ("layer_norm", _mut_unbiased_var),
    ("gelu", _mut_tanh_gelu),
])
def test_planted_mistakes_are_caught_batched(monkeypatch, target, mut):
    monkeypatch.setattr(ofw, target, mut)
    shape = tiny_shape(B=2, S=8, D=16, H=2, F_=32, L=2, causal=False)
    prm = synth.params(12, shape, ln_affine="random", bias_std=0.3)
    x = synth.input_x(12, shape) * np.float32(2.0)
    lens = np.array([8, 6], dtype=np.int32)
    ours = ofw.forward_batched(prm, 2, x, lens, False)
    ref = _torch_forward(prm, shape, x, lens, False, norm_first=True)
    diff = max(np.max(np.abs(ours[b, :lens[b]] - ref[b, :lens[b]])) for b in range(2))
    assert diff > 1e-6, f"mutation {mut.__name__} not caught (diff {diff})"
