"""GPU parity of the single-pass block draft and of context injection.

Tolerance: max relative error <= 1e-2 (max |gpu - oracle| / max |oracle|)
for bf16-path hidden states and logits; top-k is compared with the same
tolerance (an id is correct if its oracle logit is within 1e-2 * max|logit|
of the oracle's k-th value).  The oracle runs in float64 on the same
bf16-rounded weights and inputs."""

import numpy as np
import pytest
import torch

import block_speculative_decoding_ctx_gb300 as dfl
import dflash_testutil as tu
from block_speculative_decoding_ctx_gb300 import synth
from oracle import model as om
from oracle import sampling as osamp

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dfl.lib()


CASES = [
    # name, B, gamma, context lengths (window of tiny = 64, small = 256, small128 = 512)
    ("tiny", 2, 4, [64, 30]),
    ("tiny", 3, 4, [0, 1, 65]),
    ("small", 3, 8, [300, 256, 17]),
    # head dim 64 with ragged, empty and wrapped windows
    ("tiny", 4, 4, [64, 30, 0, 200]),
    ("small", 5, 8, [300, 256, 17, 0, 1000]),
    ("small128", 2, 16, [512, 700]),
    ("small128", 4, 8, [100, 513, 1, 2000]),
    # 17-32 tokens: RMSNorm folded into the GEMMs, split-K through clusters
    ("small", 4, 8, [300, 17, 256, 1000]),
    ("small128", 3, 8, [100, 513, 2000]),
    # 64-token tiles with enough weight tiles for the single-CTA persistent kernel
    ("wide", 8, 8, [300] * 4 + [17, 256, 0, 1000]),
    ("wide", 16, 8, [256] * 8 + [10, 300, 40, 999, 257, 255, 1, 0]),
    ("wide", 32, 8, [300] * 32),
    ("wide", 20, 16, [180] * 20),
]


@pytest.mark.parametrize("name,B,gamma,lens", CASES)
def test_draft_block_matches_oracle(name, B, gamma, lens):
    dims = synth.DIMS[name]
    W = synth.weights(dims, 11, random_gains=True)
    rk, rv = synth.ring(dims, B, 12)
    anchor = synth.token_ids(B, dims["vocab"], 13)
    L = torch.tensor(lens, dtype=torch.int64)
    ref = om.draft_pass(tu.oracle_cfg(dims), W, rk, rv, L.numpy(), anchor.numpy(), gamma)
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=B, gamma_max=max(gamma, 8)), tu.to_dev(W))
    got = tu.run_draft(h, anchor, L, rk.cuda(), rv.cuda(), gamma, topk=4)
    want = ref["logits"].reshape(B, gamma - 1, -1)
    assert tu.rel_err(got["logits"], want) <= TOL
    flat = want.reshape(-1, want.shape[-1])
    tu.check_topk(got["topk_ids"].reshape(-1, 4), got["topk_vals"].reshape(-1, 4), flat, TOL)
    lse = om.logsumexp(flat)
    assert np.abs(got["lse"].reshape(-1) - lse).max() <= TOL * np.abs(flat).max()
    np.testing.assert_array_equal(got["draft"], got["topk_ids"][..., 0])


def test_draft_block_at_the_largest_query_group_matches_oracle():
    """128 query rows per KV head, the largest a configuration may have: 8
    query heads per KV head at gamma 16, so every tensor-memory lane quarter
    of the attention holds query rows (contexts 300 and 7: a split with a
    partly visible last tile, and one with only part of a tile)."""
    dims = dict(synth.DIMS["small"], n_q=16, n_kv=2)
    B, gamma = 2, 16
    W = synth.weights(dims, 21, random_gains=True)
    rk, rv = synth.ring(dims, B, 22)
    anchor = synth.token_ids(B, dims["vocab"], 23)
    L = torch.tensor([300, 7], dtype=torch.int64)
    ref = om.draft_pass(tu.oracle_cfg(dims), W, rk, rv, L.numpy(), anchor.numpy(), gamma)
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=B, gamma_max=gamma), tu.to_dev(W))
    got = tu.run_draft(h, anchor, L, rk.cuda(), rv.cuda(), gamma, topk=4)
    want = ref["logits"].reshape(B, gamma - 1, -1)
    assert tu.rel_err(got["logits"], want) <= TOL


def test_draft_block_long_window_at_small_batch_matches_oracle():
    """A long window at small batch: every KV head's keys split over a full
    cluster of CTAs merged through distributed shared memory.  Contexts 2000,
    700, 100 and 0 leave some splits without keys."""
    dims = dict(synth.DIMS["small"], window=2048)
    B, gamma = 4, 8
    W = synth.weights(dims, 18, random_gains=True)
    rk, rv = synth.ring(dims, B, 19)
    anchor = synth.token_ids(B, dims["vocab"], 20)
    L = torch.tensor([2000, 700, 100, 0], dtype=torch.int64)
    ref = om.draft_pass(tu.oracle_cfg(dims), W, rk, rv, L.numpy(), anchor.numpy(), gamma)
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=B, gamma_max=gamma), tu.to_dev(W))
    dev = torch.device("cuda")
    ws = dfl.workspace(dfl.dflash_draft_workspace_bytes(h))
    for _ in range(2):                    # one workspace, reused
        logits = torch.full((B, gamma - 1, dims["vocab"]), -7.0, device=dev)
        dfl.dflash_draft_block(h, anchor.to(dev), L.to(dev), rk.cuda(), rv.cuda(), gamma, ws,
                               out=dict(logits=logits))
        torch.cuda.synchronize()
        assert dfl.dflash_read_status(ws) == 0
        assert tu.rel_err(logits.cpu().numpy(), ref["logits"]) <= TOL


@pytest.mark.parametrize("name,B,gamma,lens,k", [("small", 3, 8, [300, 17, 0], 4),
                                                  ("wide", 32, 8, [300] * 31 + [40], 4),
                                                  ("small128", 2, 16, [512, 3], 16)])
def test_topk_without_logits_matches_oracle(name, B, gamma, lens, k):
    """No logits requested: top-k, log-sum-exp and the top-1 draft come from
    the LM head's per-tile partials alone (the fp32 logits are never written)."""
    dims = synth.DIMS[name]
    W = synth.weights(dims, 15, random_gains=True)
    rk, rv = synth.ring(dims, B, 16)
    anchor = synth.token_ids(B, dims["vocab"], 17)
    L = torch.tensor(lens, dtype=torch.int64)
    ref = om.draft_pass(tu.oracle_cfg(dims), W, rk, rv, L.numpy(), anchor.numpy(), gamma)
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=B, gamma_max=max(gamma, 8), topk_max=k), tu.to_dev(W))
    got = tu.run_draft(h, anchor, L, rk.cuda(), rv.cuda(), gamma, topk=k, with_logits=False)
    flat = ref["logits"].reshape(-1, ref["logits"].shape[-1])
    tu.check_topk(got["topk_ids"].reshape(-1, k), got["topk_vals"].reshape(-1, k), flat, TOL)
    assert np.abs(got["lse"].reshape(-1) - om.logsumexp(flat)).max() <= TOL * np.abs(flat).max()
    np.testing.assert_array_equal(got["draft"], got["topk_ids"][..., 0])


def test_draft_block_with_request_slots_and_topk16():
    dims = synth.DIMS["small"]
    B, gamma = 2, 8
    W = synth.weights(dims, 21, random_gains=True)
    rk, rv = synth.ring(dims, 4, 22)                  # ring rows 0..3
    slots = torch.tensor([3, 1], dtype=torch.int32)
    anchor = synth.token_ids(B, dims["vocab"], 23)
    L = torch.tensor([400, 90], dtype=torch.int64)
    ref = om.draft_pass(tu.oracle_cfg(dims), W, rk[:, [3, 1]], rv[:, [3, 1]], L.numpy(),
                        anchor.numpy(), gamma)
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=B, gamma_max=gamma, topk_max=16), tu.to_dev(W))
    got = tu.run_draft(h, anchor, L, rk.cuda(), rv.cuda(), gamma, topk=16, req_slot=slots.cuda())
    want = ref["logits"]
    assert tu.rel_err(got["logits"], want) <= TOL
    tu.check_topk(got["topk_ids"].reshape(-1, 16), got["topk_vals"].reshape(-1, 16),
                  want.reshape(-1, want.shape[-1]), TOL)


@pytest.mark.parametrize("name,B,gamma,lens", [("small", 3, 8, [256, 40, 999]),
                                                ("small128", 4, 16, [512, 0, 7, 2000])])
def test_sampled_draft_then_sampled_verify_chain(name, B, gamma, lens):
    """draft_block with T = 0.7, top-p 0.99 gives q and y ~ q; stand-in
    target logits (draft logits + N(0, 1)) give p through dflash_probs; the
    sampled verification of y is bit-exact against the oracle fed the same
    float32 p, q and y.  q is checked against the sampling preparation of the
    drafter's own logits (1e-5) and against the oracle's logits within the
    bound those logits' error implies."""
    from oracle import verify as over
    dims = synth.DIMS[name]
    T, top_p, step = 0.7, 0.99, 5
    G, V = gamma - 1, dims["vocab"]
    W = synth.weights(dims, 31, random_gains=True)
    rk, rv = synth.ring(dims, B, 32)
    anchor = synth.token_ids(B, V, 33)
    L = torch.tensor(lens, dtype=torch.int64)
    seeds = synth.seeds(B, 34)
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=B, gamma_max=gamma), tu.to_dev(W))
    sp = dict(temperature=T, top_p=top_p, seeds=seeds.cuda(), step=step)
    got = tu.run_draft(h, anchor, L, rk.cuda(), rv.cuda(), gamma, topk=4, sampling=sp)
    ref = om.draft_pass(tu.oracle_cfg(dims), W, rk, rv, L.numpy(), anchor.numpy(), gamma)
    z = got["logits"]
    assert tu.rel_err(z, ref["logits"]) <= TOL
    tu.check_probs(got["q"], osamp.probs(z, T, top_p))
    tu.check_q_against_oracle_logits(got["q"], z, ref["logits"], T, top_p)
    seeds_u = seeds.numpy().view(np.uint64)
    np.testing.assert_array_equal(got["draft"], osamp.draft_draw(got["q"], seeds_u, step))

    t = (np.concatenate([z, z[:, G - 1:]], axis=1) +
         synth.normal((B, gamma, V), 1.0, 35).numpy()).astype(np.float32)
    dev = torch.device("cuda")
    tt = torch.from_numpy(t).to(dev)
    p = torch.empty_like(tt)
    dfl.dflash_probs(tt, T, top_p, p, dfl.workspace(dfl.dflash_probs_workspace_bytes(B * gamma, V)))
    n = torch.full((B,), -7, dtype=torch.int32, device=dev)
    tok = torch.full((B, gamma), -7, dtype=torch.int32, device=dev)
    ws_v = dfl.workspace(dfl.dflash_verify_workspace_bytes(B, gamma, V))
    dfl.dflash_verify(dfl.DFLASH_VERIFY_SAMPLED, p, torch.from_numpy(got["draft"]).to(dev), n, tok,
                      ws_v, q=torch.from_numpy(got["q"]).to(dev), seeds=seeds.cuda(), step=step)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws_v) == 0
    p_np = p.cpu().numpy()
    tu.check_probs(p_np, osamp.probs(t, T, top_p))
    want_n, want_tok = over.sampled(p_np, got["q"], got["draft"], seeds_u, step)
    np.testing.assert_array_equal(n.cpu().numpy(), want_n)
    np.testing.assert_array_equal(tok.cpu().numpy(), want_tok)


@pytest.mark.parametrize("B,G,V", [(1, 7, 1024), (5, 3, 5003), (4, 15, 151936)])
def test_sample_draft_bit_exact(B, G, V):
    logits = synth.normal((B, G, V), 2.0, 40 + B).numpy()
    q = osamp.probs(logits, 0.7, 0.99).astype(np.float32)
    seeds = synth.seeds(B, 41).numpy().view(np.uint64)
    want = osamp.draft_draw(q, seeds, 77)
    y = torch.full((B, G), -7, dtype=torch.int32, device="cuda")
    ws = dfl.workspace(dfl.dflash_sample_workspace_bytes(B * G, V))
    for _ in range(2):
        dfl.dflash_sample_draft(torch.from_numpy(q).cuda(), torch.from_numpy(seeds.view(np.int64)).cuda(),
                                77, y, ws)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(y.cpu().numpy(), want)


# ------------------------------------------------------------ ctx_append

def _oracle_ring(dims, W, B, feats, starts, n_new):
    shape = (dims["n_layers"], B, dims["n_kv"], dims["window"], dims["hd"])
    rk, rv = np.zeros(shape), np.zeros(shape)
    cfg = tu.oracle_cfg(dims)
    for b in range(B):
        if n_new[b]:
            om.ctx_append(cfg, W, rk, rv, b, feats[b, :n_new[b]], int(starts[b]))
    return rk, rv


@pytest.mark.parametrize("name,B,n_max,starts,n_new", [
    ("tiny", 2, 8, [0, 61], [8, 5]),          # second request wraps the window
    ("small", 3, 40, [5, 250, 1000], [40, 17, 0]),
    ("small128", 2, 20, [511, 3], [20, 1]),
    # up to 32 tokens the RMSNorm is folded into the W_c and K/V GEMMs
    ("small128", 2, 16, [511, 3], [16, 9]),
    ("small", 4, 8, [0, 255, 1000, 7], [8, 1, 0, 5]),
])
def test_ctx_append_matches_oracle(name, B, n_max, starts, n_new):
    dims = synth.DIMS[name]
    W = synth.weights(dims, 51, random_gains=True)
    feats = synth.features(dims, B * n_max, 52).reshape(B, n_max, dims["n_feat"], dims["feat_dim"])
    want_k, want_v = _oracle_ring(dims, W, B, feats, starts, n_new)
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=B, gamma_max=8, append_max=n_max), tu.to_dev(W))
    shape = (dims["n_layers"], B, dims["n_kv"], dims["window"], dims["hd"])
    rk = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    rv = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    ctx = torch.tensor(starts, dtype=torch.int64, device="cuda")
    nn = torch.tensor(n_new, dtype=torch.int32, device="cuda")
    ws = dfl.workspace(dfl.dflash_append_workspace_bytes(h))
    dfl.dflash_ctx_append(h, feats.cuda(), nn, ctx, rk, rv, ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    assert ctx.cpu().tolist() == [s + n for s, n in zip(starts, n_new)]
    gk, gv = rk.float().cpu().numpy(), rv.float().cpu().numpy()
    written = np.abs(want_k).sum(axis=(0, 2, 4)) > 0          # [B, W] slots written
    assert ((gk != 0).any(axis=(0, 2, 4)) == written).all()   # nothing else touched
    assert tu.rel_err(gk, want_k) <= TOL
    assert tu.rel_err(gv, want_v) <= TOL


def test_prefill_then_draft_chain_matches_oracle():
    """Long prompts: append only the last W positions (the ring wraps), then
    draft; the oracle runs the same chain."""
    dims = synth.DIMS["small"]
    Wn = dims["window"]
    B, gamma = 2, 8
    lens = [700, 100]
    W = synth.weights(dims, 61, random_gains=True)
    feats = synth.features(dims, B * Wn, 62).reshape(B, Wn, dims["n_feat"], dims["feat_dim"])
    starts = [L - min(L, Wn) for L in lens]
    n_new = [min(L, Wn) for L in lens]
    ok, ov = _oracle_ring(dims, W, B, feats, starts, n_new)
    anchor = synth.token_ids(B, dims["vocab"], 63)
    ref = om.draft_pass(tu.oracle_cfg(dims), W, ok, ov, np.array(lens), anchor.numpy(), gamma)
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=B, gamma_max=gamma, append_max=Wn), tu.to_dev(W))
    shape = (dims["n_layers"], B, dims["n_kv"], Wn, dims["hd"])
    rk = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    rv = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    ctx = torch.tensor(starts, dtype=torch.int64, device="cuda")
    ws = dfl.workspace(dfl.dflash_append_workspace_bytes(h))
    dfl.dflash_ctx_append(h, feats.cuda(), torch.tensor(n_new, dtype=torch.int32, device="cuda"), ctx,
                          rk, rv, ws)
    got = tu.run_draft(h, anchor, ctx.cpu(), rk, rv, gamma, topk=4)
    assert ctx.cpu().tolist() == lens
    assert tu.rel_err(got["logits"], ref["logits"]) <= TOL
