"""GPU parity at the full drafter dimensions (5 layers, hidden 5120, 40 q /
8 KV heads of dim 128, SwiGLU 17,408, vocabulary 151,936, window 4,096).

* batch 1, gamma 8, top-4 (the launch configuration the benchmark's headline
  line times): the whole pass against the float64 oracle (logits, top-4,
  log-sum-exp).
* ctx_append: a prefill of 4,096 positions; ring entries of sampled positions
  against the oracle's H_t and K/V for those positions alone.
* batch 16 (log-uniform contexts 512 .. 131,072 capped at the window, some
  windows partly empty), batch 32 at gamma 8 and batch 32 at gamma 16 with
  top-16 (the CTA-pair GEMMs, the two-token-tile QKV, the converter-warp
  attention): logits, top-k and log-sum-exp of EVERY request.
* the sampled chain of the batch-16 configuration: draft_block with
  temperature 0.7 and top-p 0.99 (q and y ~ q), p from stand-in target logits
  (draft logits + N(0, 1)), sampled verification; accept lengths and tokens
  bit-exact against the oracle fed the same float32 p, q and y.
Tolerance 1e-2 normwise for logits, 1e-5 for float32 probabilities."""

import numpy as np
import pytest
import torch

import block_speculative_decoding_ctx_gb300 as dfl
import dflash_testutil as tu
from block_speculative_decoding_ctx_gb300 import synth
from oracle import model as om
from oracle import sampling as osamp
from oracle import verify as over

pytestmark = pytest.mark.gpu
TOL = 1e-2
DIMS = synth.DIMS["full"]


@pytest.fixture(scope="module")
def full():
    dfl.lib()
    W = synth.weights(DIMS, 7)
    return W, tu.to_dev(W), tu.widen(W)


def _check_pass(got, ref_logits, k):
    """logits, top-k and log-sum-exp of every request of a draft pass."""
    want = ref_logits
    assert tu.rel_err(got["logits"], want) <= TOL
    flat = want.reshape(-1, want.shape[-1])
    tu.check_topk(got["topk_ids"].reshape(-1, k), got["topk_vals"].reshape(-1, k), flat, TOL)
    assert np.abs(got["lse"].reshape(-1) - om.logsumexp(flat)).max() <= TOL * np.abs(flat).max()
    np.testing.assert_array_equal(got["draft"], got["topk_ids"][..., 0])


def _draft_vs_oracle(full, B, gamma, lens, k, seed):
    W, Wd, W64 = full
    rk, rv = synth.ring(DIMS, B, seed, std=1.4)
    anchor = synth.token_ids(B, DIMS["vocab"], seed + 1)
    L = torch.as_tensor(lens, dtype=torch.int64)
    h = dfl.dflash_create(tu.lib_cfg(DIMS, batch_max=B, gamma_max=gamma, topk_max=max(k, 4)), Wd)
    got = tu.run_draft(h, anchor, L, rk.cuda(), rv.cuda(), gamma, topk=k)
    ref = om.draft_pass(tu.oracle_cfg(DIMS), W64, rk.double().numpy(), rv.double().numpy(),
                        L.numpy(), anchor.numpy(), gamma)
    _check_pass(got, ref["logits"], k)


def test_full_dims_batch1_draft_matches_oracle(full):
    _draft_vs_oracle(full, 1, 8, [4096], 4, 70)


def test_full_dims_prefill_ring_entries_match_oracle(full):
    W, Wd, W64 = full
    B, n = 1, 4096
    h = dfl.dflash_create(tu.lib_cfg(DIMS, batch_max=B, gamma_max=8, append_max=n), Wd)
    feats = synth.features(DIMS, n, 72).reshape(B, n, DIMS["n_feat"], DIMS["feat_dim"])
    shape = (DIMS["n_layers"], B, DIMS["n_kv"], DIMS["window"], DIMS["hd"])
    rk = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    rv = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    start = 131072 - n                        # a long prompt: only the last W positions
    ctx = torch.tensor([start], dtype=torch.int64, device="cuda")
    ws = dfl.workspace(dfl.dflash_append_workspace_bytes(h))
    dfl.dflash_ctx_append(h, feats.cuda(), torch.tensor([n], dtype=torch.int32, device="cuda"), ctx,
                          rk, rv, ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    assert ctx.item() == start + n
    cfg = tu.oracle_cfg(DIMS)
    rows = np.array([0, 1, 777, 2048, 4094, 4095])
    H = om.fuse_features(cfg, W64, feats[0, rows])
    Ks, Vs = om.context_kv(cfg, W64, H, start + rows)
    gk, gv = rk.float().cpu().numpy(), rv.float().cpu().numpy()
    slots = (start + rows) % DIMS["window"]
    for l in range(DIMS["n_layers"]):
        assert tu.rel_err(gk[l, 0][:, slots].transpose(1, 0, 2), Ks[l]) <= TOL
        assert tu.rel_err(gv[l, 0][:, slots].transpose(1, 0, 2), Vs[l]) <= TOL


def test_full_dims_batch16_every_request(full):
    """Contexts log-uniform in 512 .. 131,072 (the ring holds the last 4,096);
    one request pinned to 0 (the block alone) and one to 700 (a partly empty
    window)."""
    lens = synth.log_uniform_lengths(16, 512, 131072, 80)
    lens[3], lens[9] = 0, 700
    _draft_vs_oracle(full, 16, 8, lens, 4, 81)


def test_full_dims_batch32_gamma8_every_request(full):
    """256 tokens: the QKV GEMM takes two 128-token tiles per weight tile (no
    K split), gate|up and the LM head the CTA-pair persistent kernel."""
    lens = torch.full((32,), 8192, dtype=torch.int64)
    lens[5], lens[17], lens[30] = 300, 0, 4095
    _draft_vs_oracle(full, 32, 8, lens, 4, 91)


def test_full_dims_batch32_gamma16_every_request_top16(full):
    """512 tokens (two 256-token tiles), the training block size and the
    top-16 candidate list: CTA-pair GEMMs on every projection with many weight
    tiles, attention with four row tiles (the converter warp)."""
    lens = torch.full((32,), 8192, dtype=torch.int64)
    lens[0], lens[11], lens[20], lens[31] = 1, 300, 4096, 0
    _draft_vs_oracle(full, 32, 16, lens, 16, 101)


def test_full_dims_batch16_sampled_chain(full):
    """Draft with sampling (T = 0.7, top-p 0.99), stand-in target logits =
    draft logits + N(0, 1), p by dflash_probs, sampled verification."""
    W, Wd, W64 = full
    B, gamma, T, top_p, step = 16, 8, 0.7, 0.99, 11
    G, V = gamma - 1, DIMS["vocab"]
    lens = synth.log_uniform_lengths(B, 512, 131072, 110)
    rk, rv = synth.ring(DIMS, B, 111, std=1.4)
    anchor = synth.token_ids(B, V, 112)
    seeds = synth.seeds(B, 113)
    h = dfl.dflash_create(tu.lib_cfg(DIMS, batch_max=B, gamma_max=gamma), Wd)
    sp = dict(temperature=T, top_p=top_p, seeds=seeds.cuda(), step=step)
    got = tu.run_draft(h, anchor, lens, rk.cuda(), rv.cuda(), gamma, topk=4, sampling=sp)
    ref = om.draft_pass(tu.oracle_cfg(DIMS), W64, rk.double().numpy(), rv.double().numpy(),
                        lens.numpy(), anchor.numpy(), gamma)
    z = got["logits"]
    assert tu.rel_err(z, ref["logits"]) <= TOL
    # q is the sampling preparation of the drafter's own float32 logits, and
    # follows the oracle's logits within the bound they imply
    tu.check_probs(got["q"], osamp.probs(z, T, top_p))
    tu.check_q_against_oracle_logits(got["q"], z, ref["logits"], T, top_p)
    seeds_u = seeds.numpy().view(np.uint64)
    np.testing.assert_array_equal(got["draft"], osamp.draft_draw(got["q"], seeds_u, step))

    # stand-in target: draft logits + N(0, 1), the last row repeated for the bonus
    noise = synth.normal((B, gamma, V), 1.0, 114).numpy()
    t = np.concatenate([z, z[:, G - 1:]], axis=1) + noise
    t = t.astype(np.float32)
    dev = torch.device("cuda")
    tt = torch.from_numpy(t).to(dev)
    p = torch.empty_like(tt)
    ws_p = dfl.workspace(dfl.dflash_probs_workspace_bytes(B * gamma, V))
    dfl.dflash_probs(tt, T, top_p, p, ws_p)
    torch.cuda.synchronize()
    p_np = p.cpu().numpy()
    tu.check_probs(p_np, osamp.probs(t, T, top_p))
    n = torch.full((B,), -7, dtype=torch.int32, device=dev)
    tok = torch.full((B, gamma), -7, dtype=torch.int32, device=dev)
    ws_v = dfl.workspace(dfl.dflash_verify_workspace_bytes(B, gamma, V))
    dfl.dflash_verify(dfl.DFLASH_VERIFY_SAMPLED, p, torch.from_numpy(got["draft"]).to(dev), n, tok,
                      ws_v, q=torch.from_numpy(got["q"]).to(dev), seeds=seeds.cuda(), step=step)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws_v) == 0
    want_n, want_tok = over.sampled(p_np, got["q"], got["draft"], seeds_u, step)
    np.testing.assert_array_equal(n.cpu().numpy(), want_n)
    np.testing.assert_array_equal(tok.cpu().numpy(), want_tok)
