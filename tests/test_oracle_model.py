"""Pins of the oracle's drafter arithmetic.

Checks against closed forms, invariants and library routines (torch float64
scaled-dot-product attention, rms_norm, silu, complex rotation), never against
a retyped copy of the oracle's own formulas.

Sources: "DFlash vs DFlash 2" blog, sections "DFlash: generate the block all
at once" and "Conditioning on the target model"; model card
"Beam-1.0-501B-A23B-DFlash2", section "Model".
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import expit, logsumexp as sp_lse

from block_speculative_decoding_ctx_gb300 import synth
from oracle import model as om


def cfg_of(name, **kw):
    d = dict(synth.DIMS[name])
    d.update(kw)
    return om.Config(**d)


# -------------------------------------------------------------- primitives

def test_rmsnorm_closed_form_on_constant_vector():
    g = np.linspace(0.5, 1.5, 16)
    for c in (0.0, 1e-4, 0.3, -2.0, 7.0):
        y = om.rmsnorm(np.full(16, c), g, 1e-6)
        np.testing.assert_allclose(y, g * c / np.sqrt(c * c + 1e-6), rtol=1e-14, atol=0)


def test_rmsnorm_matches_torch_rms_norm():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(4, 96)) * 3
    g = rng.normal(size=96)
    want = F.rms_norm(torch.tensor(x), (96,), torch.tensor(g), eps=1e-6).numpy()
    np.testing.assert_allclose(om.rmsnorm(x, g, 1e-6), want, rtol=1e-12)


def test_silu_points():
    x = np.array([-30.0, -1.0, 0.0, 0.5, 3.0])
    np.testing.assert_allclose(om.silu(x), x * expit(x), rtol=1e-14)
    assert om.silu(np.array([0.0]))[0] == 0.0


def test_rope_is_complex_rotation_of_half_pairs():
    rng = np.random.default_rng(1)
    hd, theta = 64, 1.0e6
    x = rng.normal(size=(3, 2, hd))
    pos = np.array([0, 17, 100_000])
    y = om.rope(x, pos, theta)
    j = np.arange(hd // 2)
    zc = (x[..., :hd // 2] + 1j * x[..., hd // 2:]) * np.exp(
        1j * pos[:, None, None] * theta ** (-2.0 * j / hd))
    np.testing.assert_allclose(y[..., :hd // 2], zc.real, atol=1e-12)
    np.testing.assert_allclose(y[..., hd // 2:], zc.imag, atol=1e-12)
    np.testing.assert_allclose(om.rope(x, np.zeros(3), theta), x, atol=0)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(2)
    q = rng.normal(size=(1, 128))
    k = rng.normal(size=(1, 128))
    s1 = (om.rope(q, 40, 1e6) * om.rope(k, 13, 1e6)).sum()
    s2 = (om.rope(q, 1040, 1e6) * om.rope(k, 1013, 1e6)).sum()
    assert abs(s1 - s2) < 1e-9


def test_topk_and_logsumexp_against_brute_force_and_scipy():
    rng = np.random.default_rng(3)
    z = np.round(rng.normal(size=(6, 200)), 1)         # many ties
    ids, vals = om.topk(z, 5)
    for r in range(6):
        want = sorted(range(200), key=lambda i: (-z[r, i], i))[:5]
        assert ids[r].tolist() == want
        assert vals[r].tolist() == [z[r, i] for i in want]
    np.testing.assert_allclose(om.logsumexp(z), sp_lse(z, axis=-1), rtol=1e-14)


def test_drafter_parameter_count_against_model_card():
    """Model card "Beam-1.0-501B-A23B-DFlash2", section "Model": 1.93B
    parameters.  The matrices the drafter owns (5 layers + W_c; embedding and
    LM head are shared with the target) come to 1,782,579,200, below the
    card's figure by the size of the DFlash 2 modules that are out of scope."""
    n = om.drafter_matrix_params(cfg_of("full"))
    assert n == 1_782_579_200
    assert 0.90 * 1.93e9 < n < 1.93e9


# ------------------------------------------------------- feature injection

def test_fusion_with_identity_selector_is_rmsnorm_of_first_layer():
    cfg = cfg_of("tiny")
    W = synth.weights(synth.DIMS["tiny"], 1, random_gains=True)
    d = cfg.d
    wc = torch.zeros(d, cfg.n_feat * cfg.feat_dim)
    wc[:, :d] = torch.eye(d)
    W["w_c"] = wc
    feats = synth.features(synth.DIMS["tiny"], 5, 3, torch.float32).numpy()
    H = om.fuse_features(cfg, W, feats)
    want = F.rms_norm(torch.tensor(feats[:, 0, :], dtype=torch.float64), (d,),
                      W["g_c"].double(), eps=cfg.eps).numpy()
    np.testing.assert_allclose(H, want, rtol=1e-12)


def test_ring_wrap_equals_appending_only_the_last_window():
    cfg = cfg_of("tiny")
    dims = synth.DIMS["tiny"]
    W = synth.weights(dims, 2)
    L = 150                                         # > 2 windows of 64
    feats = synth.features(dims, L, 4, torch.float32).numpy()
    shape = (cfg.n_layers, 1, cfg.n_kv, cfg.window, cfg.hd)
    rk1, rv1 = np.zeros(shape), np.zeros(shape)
    for s in range(0, L, 37):                       # ragged appends
        om.ctx_append(cfg, W, rk1, rv1, 0, feats[s:s + 37], s)
    rk2, rv2 = np.zeros(shape), np.zeros(shape)
    om.ctx_append(cfg, W, rk2, rv2, 0, feats[L - cfg.window:], L - cfg.window)
    np.testing.assert_allclose(rk1, rk2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(rv1, rv2, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------- block attention

def _sdpa(q, keys, vals, visible, n_q, n_kv):
    """Library attention: q [G, Hq, hd], keys/vals [N, Hkv, hd], visible [N]."""
    tq = torch.tensor(q).permute(1, 0, 2)[None]            # [1, Hq, G, hd]
    tk = torch.tensor(keys).permute(1, 0, 2)[None]
    tv = torch.tensor(vals).permute(1, 0, 2)[None]
    mask = torch.tensor(visible)[None, None, None, :].expand(1, n_q, q.shape[0], keys.shape[0])
    o = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, enable_gqa=(n_q != n_kv))
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("L", [10, 64, 200])
@pytest.mark.parametrize("heads", [(4, 2), (4, 4), (10, 2)])
def test_block_attention_matches_library_attention(L, heads):
    n_q, n_kv = heads
    cfg = cfg_of("tiny", n_q=n_q, n_kv=n_kv)
    rng = np.random.default_rng(L + n_q)
    G = 4
    q = rng.normal(size=(G, n_q, cfg.hd))
    kb = rng.normal(size=(G, n_kv, cfg.hd))
    vb = rng.normal(size=(G, n_kv, cfg.hd))
    rk = rng.normal(size=(n_kv, cfg.window, cfg.hd))
    rv = rng.normal(size=(n_kv, cfg.window, cfg.hd))
    got = om.block_attention(cfg, q, kb, vb, rk, rv, L)
    n_valid = min(L, cfg.window)
    keys = np.concatenate([rk.transpose(1, 0, 2), kb], axis=0)
    vals = np.concatenate([rv.transpose(1, 0, 2), vb], axis=0)
    visible = np.concatenate([np.arange(cfg.window) < n_valid, np.ones(G, bool)])
    np.testing.assert_allclose(got, _sdpa(q, keys, vals, visible, n_q, n_kv), rtol=1e-10, atol=1e-12)


def test_block_attention_invariant_to_valid_slot_permutation_and_blind_to_invalid_slots():
    cfg = cfg_of("tiny")
    rng = np.random.default_rng(5)
    G, L = 4, 40
    q = rng.normal(size=(G, cfg.n_q, cfg.hd))
    kb, vb = rng.normal(size=(2, G, cfg.n_kv, cfg.hd))
    rk, rv = rng.normal(size=(2, cfg.n_kv, cfg.window, cfg.hd))
    base = om.block_attention(cfg, q, kb, vb, rk, rv, L)
    perm = np.concatenate([rng.permutation(L), np.arange(L, cfg.window)])
    np.testing.assert_allclose(om.block_attention(cfg, q, kb, vb, rk[:, perm], rv[:, perm], L),
                               base, rtol=1e-12)
    rk2, rv2 = rk.copy(), rv.copy()
    rk2[:, L:] = 1e3
    rv2[:, L:] = -1e3
    np.testing.assert_allclose(om.block_attention(cfg, q, kb, vb, rk2, rv2, L), base, rtol=1e-12)


def test_block_attention_is_non_causal_inside_the_block():
    cfg = cfg_of("tiny")
    rng = np.random.default_rng(6)
    G, L = 4, 64
    q = rng.normal(size=(G, cfg.n_q, cfg.hd))
    kb, vb = rng.normal(size=(2, G, cfg.n_kv, cfg.hd))
    rk, rv = rng.normal(size=(2, cfg.n_kv, cfg.window, cfg.hd))
    base = om.block_attention(cfg, q, kb, vb, rk, rv, L)
    vb2 = vb.copy()
    vb2[G - 1] += 5.0                                  # last block position
    out = om.block_attention(cfg, q, kb, vb2, rk, rv, L)
    assert np.abs(out[0] - base[0]).max() > 1e-3       # the anchor row sees it


# --------------------------------------------------------------- draft pass

def _rope_c(cfg, t, pos):
    """Rotate-half RoPE of t [n, heads, hd] at positions pos [n] as a complex
    product: (x_j + i x_{j+hd/2}) * exp(i pos theta^(-2j/hd))."""
    dd = torch.float64
    j = torch.arange(cfg.hd // 2, dtype=dd)
    pos = torch.as_tensor(np.asarray(pos), dtype=dd)
    rot = torch.polar(torch.ones(len(pos), cfg.hd // 2, dtype=dd),
                      pos[:, None] * cfg.rope_theta ** (-2.0 * j / cfg.hd))[:, None, :]
    z = torch.complex(t[..., :cfg.hd // 2], t[..., cfg.hd // 2:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def _library_kv(cfg, lw, h, pos):
    """K = RoPE(W^K h, pos) and V = W^V h of normalised rows h [n, d], with
    torch routines: the k and v row blocks of w_qkv (its rows are the q heads,
    then the k heads, then the v heads), the rotation as a complex product."""
    dd = torch.float64
    qd, kd = cfg.n_q * cfg.hd, cfg.n_kv * cfg.hd
    n = h.shape[0]
    qkv = torch.as_tensor(np.asarray(h), dtype=dd) @ lw["w_qkv"].to(dd).T
    k = _rope_c(cfg, qkv[:, qd:qd + kd].reshape(n, cfg.n_kv, cfg.hd), pos)
    v = qkv[:, qd + kd:].reshape(n, cfg.n_kv, cfg.hd)
    return k, v


def _library_draft_pass(cfg, W, ctx_k, ctx_v, L, anchor, gamma):
    """One request through the layers with torch float64 library routines
    (rms_norm, SDPA with GQA, silu, complex rotation).  ctx_k[l], ctx_v[l]
    [n, Hkv, hd] are the visible context keys and values of layer l (any
    order); the block forms its own keys and values with _library_kv."""
    dd = torch.float64
    ids = [anchor] + [cfg.mask_token] * (gamma - 1)
    x = W["embed"][ids].to(dd)
    pos = np.arange(L, L + gamma)
    qd = cfg.n_q * cfg.hd
    for l, lw in enumerate(W["layers"]):
        h = F.rms_norm(x, (cfg.d,), lw["g_attn"].to(dd), eps=cfg.eps)
        q = _rope_c(cfg, (h @ lw["w_qkv"][:qd].to(dd).T).reshape(gamma, cfg.n_q, cfg.hd), pos)
        k, v = _library_kv(cfg, lw, h, pos)
        keys = torch.cat([torch.as_tensor(ctx_k[l], dtype=dd), k])
        vals = torch.cat([torch.as_tensor(ctx_v[l], dtype=dd), v])
        o = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], keys.permute(1, 0, 2)[None],
                                           vals.permute(1, 0, 2)[None], enable_gqa=True)
        x = x + o[0].permute(1, 0, 2).reshape(gamma, qd) @ lw["w_o"].to(dd).T
        h = F.rms_norm(x, (cfg.d,), lw["g_mlp"].to(dd), eps=cfg.eps)
        x = x + (F.silu(h @ lw["w_gate"].to(dd).T) * (h @ lw["w_up"].to(dd).T)) @ lw["w_down"].to(dd).T
    hf = F.rms_norm(x, (cfg.d,), W["g_final"].to(dd), eps=cfg.eps)
    return (hf[1:] @ W["lm_head"].to(dd).T).numpy()


def _ring_context(cfg, rk, rv, L):
    """Visible context of request 0 of a ring: slots 0 .. min(L, W) - 1."""
    n_valid = min(L, cfg.window)
    return ([rk[l, 0].to(torch.float64).permute(1, 0, 2)[:n_valid] for l in range(cfg.n_layers)],
            [rv[l, 0].to(torch.float64).permute(1, 0, 2)[:n_valid] for l in range(cfg.n_layers)])


@pytest.mark.parametrize("L", [30, 64, 500])
def test_draft_pass_matches_library_layers(L):
    dims = dict(synth.DIMS["tiny"], n_layers=2)
    cfg = om.Config(**dims)
    W = synth.weights(dims, 3, random_gains=True)
    rk, rv = synth.ring(dims, 1, 4)
    gamma = 4
    got = om.draft_pass(cfg, W, rk, rv, [L], [17], gamma)["logits"][0]
    want = _library_draft_pass(cfg, W, *_ring_context(cfg, rk, rv, L), L, 17, gamma)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-11)


def test_draft_pass_without_attention_and_mlp_outputs_reduces_to_embedding_head():
    """With W_o = W_down = 0 the residual stream is the block embedding, so
    every MASK row gets logits = RMSNorm(embed[MASK]) W_lm^T."""
    dims = synth.DIMS["tiny"]
    cfg = om.Config(**dims)
    W = synth.weights(dims, 5, random_gains=True)
    for lw in W["layers"]:
        lw["w_o"] = torch.zeros_like(lw["w_o"])
        lw["w_down"] = torch.zeros_like(lw["w_down"])
    rk, rv = synth.ring(dims, 1, 6)
    out = om.draft_pass(cfg, W, rk, rv, [64], [3], 4)["logits"][0]
    e = W["embed"][cfg.mask_token].double()
    want = (F.rms_norm(e, (cfg.d,), W["g_final"].double(), eps=cfg.eps) @ W["lm_head"].double().T).numpy()
    for r in range(3):
        np.testing.assert_allclose(out[r], want, rtol=1e-10, atol=1e-12)


def test_draft_rows_differ_through_positions():
    """Identical MASK inputs give distinct rows only through positions."""
    dims = synth.DIMS["tiny"]
    cfg = om.Config(**dims)
    W = synth.weights(dims, 7)
    rk, rv = synth.ring(dims, 1, 8)
    out = om.draft_pass(cfg, W, rk, rv, [64], [3], 4)["logits"][0]
    assert np.abs(out[0] - out[1]).max() > 1e-6


# ------------------------------------- context K/V: the injection equation
#
# "DFlash vs DFlash 2", section "Conditioning on the target model": the keys
# and values of layer i are K_i = [W^K_i H_t ; W^K_i H_d] and
# V_i = [W^V_i H_t ; W^V_i H_d] — the context half is projected by the same
# W^K_i / W^V_i as the block half.  With rotary positions (a reading the pages
# leave open) a context key is rotated at its own absolute position exactly
# like a block key.

@pytest.mark.parametrize("dims_name", ["tiny", "small"])
def test_context_kv_is_the_blocks_key_value_projection(dims_name):
    dims = dict(synth.DIMS[dims_name], n_layers=2)
    cfg = om.Config(**dims)
    W = synth.weights(dims, 11, random_gains=True)
    rng = np.random.default_rng(11)
    H = rng.normal(size=(7, cfg.d))
    pos = np.array([0, 1, 63, 64, 1000, 65_537, 131_071])
    Ks, Vs = om.context_kv(cfg, W, H, pos)
    assert len(Ks) == len(Vs) == cfg.n_layers
    for l, lw in enumerate(W["layers"]):
        k, v = _library_kv(cfg, lw, H, pos)
        np.testing.assert_allclose(Ks[l], k.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(Vs[l], v.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("L", [5, 64, 100])
def test_appended_context_drafts_like_a_library_pass_over_projected_features(L):
    """ctx_append (fusion, projection, rotation, ring slot pos mod W) followed
    by the draft pass equals a library pass whose context keys and values are
    the block's own projection routine applied to H_t = RMSNorm(W_c concat(H))
    at positions 0 .. L-1 (the last W of them visible)."""
    dims = dict(synth.DIMS["tiny"], n_layers=2)
    cfg = om.Config(**dims)
    W = synth.weights(dims, 12, random_gains=True)
    feats = synth.features(dims, L, 13, torch.float32).numpy()
    shape = (cfg.n_layers, 1, cfg.n_kv, cfg.window, cfg.hd)
    rk, rv = np.zeros(shape), np.zeros(shape)
    for s0 in range(0, L, 29):                         # ragged appends
        om.ctx_append(cfg, W, rk, rv, 0, feats[s0:s0 + 29], s0)
    gamma = 4
    got = om.draft_pass(cfg, W, rk, rv, [L], [17], gamma)["logits"][0]

    dd = torch.float64
    cat = torch.as_tensor(feats, dtype=dd).reshape(L, cfg.n_feat * cfg.feat_dim)
    H_t = F.rms_norm(cat @ W["w_c"].to(dd).T, (cfg.d,), W["g_c"].to(dd), eps=cfg.eps)
    vis = np.arange(max(0, L - cfg.window), L)
    ctx = [_library_kv(cfg, lw, H_t[vis], vis) for lw in W["layers"]]
    want = _library_draft_pass(cfg, W, [c[0] for c in ctx], [c[1] for c in ctx], L, 17, gamma)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-11)


def test_draft_over_appended_context_is_invariant_to_a_common_position_shift():
    """Rotary scores depend only on query position minus key position: with
    the same features filling the window at positions s0 .. s0+W-1 and the
    block at s0+W, the logits cannot depend on s0.  Context keys left
    unrotated, or rotated by another convention than the block's, break this."""
    dims = synth.DIMS["tiny"]
    cfg = om.Config(**dims)
    W = synth.weights(dims, 14, random_gains=True)
    n = cfg.window
    feats = synth.features(dims, n, 15, torch.float32).numpy()
    shape = (cfg.n_layers, 1, cfg.n_kv, cfg.window, cfg.hd)

    def logits_after(fe, s0):
        rk, rv = np.zeros(shape), np.zeros(shape)
        om.ctx_append(cfg, W, rk, rv, 0, fe, s0)
        return om.draft_pass(cfg, W, rk, rv, [s0 + n], [5], 4)["logits"][0]

    base = logits_after(feats, 0)
    for s0 in (37, 100_003):
        np.testing.assert_allclose(logits_after(feats, s0), base, rtol=1e-7, atol=1e-9)
    # the order of the context matters only through the keys' rotations:
    # without them a reversed context would give the same logits
    assert np.abs(logits_after(feats[::-1].copy(), 0) - base).max() > 1e-4
