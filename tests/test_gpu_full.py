"""GPU parity at the full drafter dimensions (5 layers, hidden 5120, 40 q /
8 KV heads of dim 128, SwiGLU 17,408, vocabulary 151,936, window 4,096), in
the launch configuration the benchmark times (batch 1, gamma 8, top-4).

* draft_block: the whole pass is compared with the float64 oracle (logits,
  top-4, log-sum-exp) on a synthetic full ring.
* ctx_append: a prefill of 4,096 positions; ring entries of sampled positions
  are compared with the oracle's H_t and K/V for those positions alone.
* the batch-16 config: ragged log-uniform contexts; one sampled request's
  draft is recomputed by the oracle.
* batch 32, gamma 8: two sampled requests (the wide-token-tile GEMM paths).
Tolerance 1e-2 normwise, as for the small shapes."""

import numpy as np
import pytest
import torch

import block_speculative_decoding_ctx_gb300 as dfl
import dflash_testutil as tu
from block_speculative_decoding_ctx_gb300 import synth
from oracle import model as om

pytestmark = pytest.mark.gpu
TOL = 1e-2
DIMS = synth.DIMS["full"]


@pytest.fixture(scope="module")
def full():
    dfl.lib()
    W = synth.weights(DIMS, 7)
    Wd = tu.to_dev(W)
    return W, Wd


def test_full_dims_batch1_draft_matches_oracle(full):
    W, Wd = full
    B, gamma = 1, 8
    rk, rv = synth.ring(DIMS, B, 70, std=1.4)
    anchor = synth.token_ids(B, DIMS["vocab"], 71)
    L = torch.tensor([4096], dtype=torch.int64)
    h = dfl.dflash_create(tu.lib_cfg(DIMS, batch_max=B, gamma_max=gamma), Wd)
    got = tu.run_draft(h, anchor, L, rk.cuda(), rv.cuda(), gamma, topk=4)
    ref = om.draft_pass(tu.oracle_cfg(DIMS), W, rk, rv, L.numpy(), anchor.numpy(), gamma)
    want = ref["logits"]
    assert tu.rel_err(got["logits"], want) <= TOL
    flat = want.reshape(-1, want.shape[-1])
    tu.check_topk(got["topk_ids"].reshape(-1, 4), got["topk_vals"].reshape(-1, 4), flat, TOL)
    assert np.abs(got["lse"].reshape(-1) - om.logsumexp(flat)).max() <= TOL * np.abs(flat).max()


def test_full_dims_prefill_ring_entries_match_oracle(full):
    W, Wd = full
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
    H = om.fuse_features(cfg, W, feats[0, rows])
    Ks, Vs = om.context_kv(cfg, W, H, start + rows)
    gk, gv = rk.float().cpu().numpy(), rv.float().cpu().numpy()
    slots = (start + rows) % DIMS["window"]
    for l in range(DIMS["n_layers"]):
        assert tu.rel_err(gk[l, 0][:, slots].transpose(1, 0, 2), Ks[l]) <= TOL
        assert tu.rel_err(gv[l, 0][:, slots].transpose(1, 0, 2), Vs[l]) <= TOL


def test_batch16_ragged_contexts_sampled_request(full):
    W, Wd = full
    B, gamma = 16, 8
    lens = synth.log_uniform_lengths(B, 512, 131072, 80)
    rk, rv = synth.ring(DIMS, B, 81, std=1.4)
    anchor = synth.token_ids(B, DIMS["vocab"], 82)
    h = dfl.dflash_create(tu.lib_cfg(DIMS, batch_max=B, gamma_max=gamma), Wd)
    got = tu.run_draft(h, anchor, lens, rk.cuda(), rv.cuda(), gamma, topk=4)
    # one request with a short context (partly empty window) and one long
    short = int(torch.argmin(lens))
    long = int(torch.argmax(lens))
    ref = om.draft_pass(tu.oracle_cfg(DIMS), W, rk, rv, lens.numpy(), anchor.numpy(), gamma,
                        requests=[short, long])
    for i, b in enumerate([short, long]):
        assert tu.rel_err(got["logits"][b], ref["logits"][i]) <= TOL


def test_batch32_gamma8_sampled_requests(full):
    """256 tokens: the QKV GEMM takes two 128-token tiles per weight tile (no
    K split), gate|up and the LM head the CTA-pair persistent kernel."""
    W, Wd = full
    B, gamma = 32, 8
    lens = torch.full((B,), 8192, dtype=torch.int64)
    lens[5] = 300                                   # one partly empty window
    rk, rv = synth.ring(DIMS, B, 91, std=1.4)
    anchor = synth.token_ids(B, DIMS["vocab"], 92)
    h = dfl.dflash_create(tu.lib_cfg(DIMS, batch_max=B, gamma_max=gamma), Wd)
    got = tu.run_draft(h, anchor, lens, rk.cuda(), rv.cuda(), gamma, topk=4)
    picks = [5, 31]
    ref = om.draft_pass(tu.oracle_cfg(DIMS), W, rk, rv, lens.numpy(), anchor.numpy(), gamma,
                        requests=picks)
    for i, b in enumerate(picks):
        assert tu.rel_err(got["logits"][b], ref["logits"][i]) <= TOL
