"""GPU checks of the cycle as a whole: graph capture, device-side commit
outputs, and device-side argument checks reported through the status word."""

import numpy as np
import pytest
import torch

import block_speculative_decoding_ctx_gb300 as dfl
import dflash_testutil as tu
from block_speculative_decoding_ctx_gb300 import synth
from oracle import verify as over

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dfl.lib()


def _setup(name="small", B=2, gamma=8):
    dims = synth.DIMS[name]
    W = synth.weights(dims, 91, random_gains=True)
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=B, gamma_max=gamma, append_max=gamma), tu.to_dev(W))
    rk, rv = synth.ring(dims, B, 92)
    return dims, h, rk.cuda(), rv.cuda()


def test_captured_cycle_replays_like_eager_calls():
    dims, h, rk, rv = _setup()
    B, gamma, V = 2, 8, dims["vocab"]
    dev = torch.device("cuda")
    feats = synth.features(dims, B * gamma, 93).reshape(B, gamma, dims["n_feat"], dims["feat_dim"]).cuda()
    noise = synth.normal((B, gamma, V), 0.05, 94).cuda()

    def state():
        return dict(ctx=torch.tensor([300, 40], dtype=torch.int64, device=dev),
                    anchor=torch.tensor([5, 7], dtype=torch.int32, device=dev),
                    n_app=torch.tensor([3, 1], dtype=torch.int32, device=dev),
                    rk=rk.clone(), rv=rv.clone(),
                    logits=torch.empty((B, gamma - 1, V), device=dev),
                    draft=torch.empty((B, gamma - 1), dtype=torch.int32, device=dev),
                    target=torch.empty((B, gamma, V), device=dev),
                    acc=torch.empty(B, dtype=torch.int32, device=dev),
                    tok=torch.empty((B, gamma), dtype=torch.int32, device=dev),
                    ws_a=dfl.workspace(dfl.dflash_append_workspace_bytes(h)),
                    ws_d=dfl.workspace(dfl.dflash_draft_workspace_bytes(h)),
                    ws_v=dfl.workspace(dfl.dflash_verify_workspace_bytes(B, gamma, V)))

    def cycle(st):
        dfl.dflash_ctx_append(h, feats, st["n_app"], st["ctx"], st["rk"], st["rv"], st["ws_a"])
        dfl.dflash_draft_block(h, st["anchor"], st["ctx"], st["rk"], st["rv"], gamma, st["ws_d"],
                               out=dict(logits=st["logits"], draft=st["draft"]))
        torch.add(st["logits"], noise[:, :gamma - 1], out=st["target"][:, :gamma - 1])
        torch.add(st["logits"][:, gamma - 2], noise[:, gamma - 1], out=st["target"][:, gamma - 1])
        dfl.dflash_verify(dfl.DFLASH_VERIFY_GREEDY, st["target"], st["draft"], st["acc"], st["tok"],
                          st["ws_v"], next_anchor=st["anchor"], n_append=st["n_app"])

    eager = state()
    hist_e = []
    for _ in range(3):
        cycle(eager)
        hist_e.append((eager["acc"].cpu().clone(), eager["tok"].cpu().clone(), eager["ctx"].cpu().clone()))

    graphed = state()
    s = torch.cuda.Stream()
    warm = state()
    with torch.cuda.stream(s):
        cycle(warm)                      # first calls outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cycle(graphed)
    # capture records work without running it: reset the state, then replay
    fresh = state()
    for k in ("ctx", "anchor", "n_app", "rk", "rv"):
        graphed[k].copy_(fresh[k])
    for ws in ("ws_a", "ws_d", "ws_v"):
        graphed[ws].zero_()
    torch.cuda.synchronize()
    for i in range(3):
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        a, t, c = hist_e[i]
        assert torch.equal(graphed["acc"].cpu(), a)
        assert torch.equal(graphed["tok"].cpu(), t)
        assert torch.equal(graphed["ctx"].cpu(), c)
    # commit outputs follow the committed tokens
    n = graphed["acc"].cpu().numpy()
    tok = graphed["tok"].cpu().numpy()
    assert (graphed["n_app"].cpu().numpy() == n + 1).all()
    assert (graphed["anchor"].cpu().numpy() == tok[np.arange(B), n]).all()


def test_captured_cycle_matches_oracle_cycle():
    """Three replays of one captured cycle (ctx_append of the positions the
    last verification committed, draft_block, greedy verify writing the next
    anchor and append count on the device) against the oracle running the
    same cycle: its own ring, context lengths and anchors.

    Before each replay the test writes the stand-in target logits (outside
    the graph), designed from the oracle's drafts for that cycle so that each
    request accepts a chosen number of drafts (all of them, with the bonus, in
    one case).  Draft tokens are compared with the oracle's top-1 wherever its
    margin exceeds twice the logit tolerance, and tolerance-aware elsewhere;
    the oracle then verifies the GPU's drafts, so accept lengths, committed
    tokens, next anchors, append counts and context lengths are compared bit
    for bit, and the ring entries appended each cycle within 1e-2."""
    from oracle import model as om
    dims, h, rk0, rv0 = _setup()
    B, gamma, V = 2, 8, dims["vocab"]
    G = gamma - 1
    TOL = 1e-2
    dev = torch.device("cuda")
    W = synth.weights(dims, 91, random_gains=True)          # the weights _setup loaded
    cfg = tu.oracle_cfg(dims)
    feats = synth.features(dims, B * gamma, 93).reshape(B, gamma, dims["n_feat"], dims["feat_dim"])
    ctx0, anchor0, napp0 = [300, 40], [5, 7], [3, 1]
    design = [(3, 0), (G, 2), (1, 5)]                       # drafts each request should accept

    def state():
        return dict(ctx=torch.tensor(ctx0, dtype=torch.int64, device=dev),
                    anchor=torch.tensor(anchor0, dtype=torch.int32, device=dev),
                    n_app=torch.tensor(napp0, dtype=torch.int32, device=dev),
                    rk=rk0.clone(), rv=rv0.clone(),
                    logits=torch.empty((B, G, V), device=dev),
                    draft=torch.empty((B, G), dtype=torch.int32, device=dev),
                    target=torch.zeros((B, gamma, V), device=dev),
                    acc=torch.empty(B, dtype=torch.int32, device=dev),
                    tok=torch.empty((B, gamma), dtype=torch.int32, device=dev),
                    ws_a=dfl.workspace(dfl.dflash_append_workspace_bytes(h)),
                    ws_d=dfl.workspace(dfl.dflash_draft_workspace_bytes(h)),
                    ws_v=dfl.workspace(dfl.dflash_verify_workspace_bytes(B, gamma, V)))

    fd = feats.cuda()

    def cycle(st):
        dfl.dflash_ctx_append(h, fd, st["n_app"], st["ctx"], st["rk"], st["rv"], st["ws_a"])
        dfl.dflash_draft_block(h, st["anchor"], st["ctx"], st["rk"], st["rv"], gamma, st["ws_d"],
                               out=dict(logits=st["logits"], draft=st["draft"]))
        dfl.dflash_verify(dfl.DFLASH_VERIFY_GREEDY, st["target"], st["draft"], st["acc"], st["tok"],
                          st["ws_v"], next_anchor=st["anchor"], n_append=st["n_app"])

    s = torch.cuda.Stream()
    warm = state()
    with torch.cuda.stream(s):
        cycle(warm)                      # first calls outside the capture
    torch.cuda.synchronize()
    st = state()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cycle(st)
    fresh = state()                      # capture recorded work without running it
    for k in ("ctx", "anchor", "n_app", "rk", "rv"):
        st[k].copy_(fresh[k])
    for ws in ("ws_a", "ws_d", "ws_v"):
        st[ws].zero_()
    torch.cuda.synchronize()

    ork, orv = rk0.double().cpu().numpy(), rv0.double().cpu().numpy()
    octx, oanc, oapp = np.array(ctx0), np.array(anchor0), np.array(napp0)
    rng = np.random.default_rng(95)
    for cyc_i, ks in enumerate(design):
        # the oracle's cycle up to its drafts
        appended = []
        for b in range(B):
            om.ctx_append(cfg, W, ork, orv, b, feats[b, :oapp[b]], int(octx[b]))
            appended.append((int(octx[b]), int(oapp[b])))
        octx = octx + oapp
        z = om.draft_pass(cfg, W, ork, orv, octx, oanc, gamma)["logits"]
        top = z.argmax(-1)
        # stand-in target designed from the oracle's drafts
        t = rng.normal(size=(B, gamma, V)).astype(np.float32)
        for b, k in enumerate(ks):
            for i in range(k):
                t[b, i, top[b, i]] = 20.0
            c = (int(top[b, k]) + 17 if k < G else 3 * cyc_i + 11) % V
            t[b, k, c] = 20.0
        st["target"].copy_(torch.from_numpy(t))
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        zg = st["logits"].cpu().numpy()
        assert tu.rel_err(zg, z) <= TOL
        scale = np.abs(z).max()
        yg = st["draft"].cpu().numpy()
        srt = np.sort(z, axis=-1)
        for b in range(B):
            for i in range(G):
                if srt[b, i, -1] - srt[b, i, -2] > 2 * TOL * scale:
                    assert yg[b, i] == top[b, i]
                else:
                    assert z[b, i, yg[b, i]] >= srt[b, i, -1] - TOL * scale
        n_o, tok_o = over.greedy(t, yg)
        np.testing.assert_array_equal(st["acc"].cpu().numpy(), n_o)
        np.testing.assert_array_equal(st["tok"].cpu().numpy(), tok_o)
        oanc = tok_o[np.arange(B), n_o].astype(np.int64)
        oapp = n_o + 1
        np.testing.assert_array_equal(st["anchor"].cpu().numpy(), oanc)
        np.testing.assert_array_equal(st["n_app"].cpu().numpy(), oapp)
        np.testing.assert_array_equal(st["ctx"].cpu().numpy(), octx)
        gk, gv = st["rk"].double().cpu().numpy(), st["rv"].double().cpu().numpy()
        for b, (p0, n) in enumerate(appended):
            slots = (p0 + np.arange(n)) % dims["window"]
            assert tu.rel_err(gk[:, b][:, :, slots], ork[:, b][:, :, slots]) <= TOL
            assert tu.rel_err(gv[:, b][:, :, slots], orv[:, b][:, :, slots]) <= TOL
    assert dfl.dflash_read_status(st["ws_a"]) == 0
    assert dfl.dflash_read_status(st["ws_d"]) == 0
    assert dfl.dflash_read_status(st["ws_v"]) == 0


def test_verify_commit_outputs_sampled():
    B, gamma, V = 5, 6, 300
    rng = np.random.default_rng(3)
    p = rng.dirichlet(np.ones(V), size=(B, gamma)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=(B, gamma - 1)).astype(np.float32)
    seeds = np.arange(B, dtype=np.uint64) + np.uint64(17)
    from oracle import sampling as osamp
    y = osamp.draft_draw(q, seeds, 4).astype(np.int32)
    n_ref, tok_ref = over.sampled(p, q, y, seeds, 4)
    dev = torch.device("cuda")
    n = torch.empty(B, dtype=torch.int32, device=dev)
    tok = torch.empty((B, gamma), dtype=torch.int32, device=dev)
    anc = torch.empty(B, dtype=torch.int32, device=dev)
    app = torch.empty(B, dtype=torch.int32, device=dev)
    ws = dfl.workspace(dfl.dflash_verify_workspace_bytes(B, gamma, V))
    dfl.dflash_verify(dfl.DFLASH_VERIFY_SAMPLED, torch.from_numpy(p).to(dev), torch.from_numpy(y).to(dev),
                      n, tok, ws, q=torch.from_numpy(q).to(dev),
                      seeds=torch.from_numpy(seeds.view(np.int64)).to(dev), step=4,
                      next_anchor=anc, n_append=app)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(n.cpu().numpy(), n_ref)
    np.testing.assert_array_equal(anc.cpu().numpy(), tok_ref[np.arange(B), n_ref])
    np.testing.assert_array_equal(app.cpu().numpy(), n_ref + 1)


def test_out_of_range_slot_and_anchor_are_reported_not_faulted():
    dims, h, rk, rv = _setup(B=2)
    B, gamma = 2, 8
    dev = torch.device("cuda")
    ws = dfl.workspace(dfl.dflash_draft_workspace_bytes(h))
    bad_slot = torch.tensor([0, 9], dtype=torch.int32, device=dev)      # ring has 2 rows
    dfl.dflash_draft_block(h, torch.tensor([1, 2], dtype=torch.int32, device=dev),
                           torch.tensor([100, 100], dtype=torch.int64, device=dev), rk, rv, gamma, ws,
                           out=dict(draft=torch.empty((B, gamma - 1), dtype=torch.int32, device=dev)),
                           req_slot=bad_slot)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == -1
    ws2 = dfl.workspace(dfl.dflash_draft_workspace_bytes(h))
    dfl.dflash_draft_block(h, torch.tensor([1, 10 ** 6], dtype=torch.int32, device=dev),
                           torch.tensor([100, 100], dtype=torch.int64, device=dev), rk, rv, gamma, ws2,
                           out=dict(draft=torch.empty((B, gamma - 1), dtype=torch.int32, device=dev)))
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws2) == -1
    # a good call afterwards still works
    ws3 = dfl.workspace(dfl.dflash_draft_workspace_bytes(h))
    dfl.dflash_draft_block(h, torch.tensor([1, 2], dtype=torch.int32, device=dev),
                           torch.tensor([100, 100], dtype=torch.int64, device=dev), rk, rv, gamma, ws3,
                           out=dict(draft=torch.empty((B, gamma - 1), dtype=torch.int32, device=dev)))
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws3) == 0


def test_host_validation_rejects_bad_draft_calls():
    dims, h, rk, rv = _setup(B=2)
    dev = torch.device("cuda")
    ws = dfl.workspace(dfl.dflash_draft_workspace_bytes(h))
    a = torch.tensor([1, 2], dtype=torch.int32, device=dev)
    L = torch.tensor([10, 10], dtype=torch.int64, device=dev)
    with pytest.raises(dfl.DflashError) as e:
        dfl.dflash_draft_block(h, a, L, rk, rv, 17, ws)                 # gamma > gamma_max
    assert e.value.code == -2
    with pytest.raises(dfl.DflashError) as e:
        dfl.dflash_draft_block(h, a, L, rk, rv, 8, ws[:1024])           # workspace too small
    assert e.value.code == -7
    with pytest.raises(dfl.DflashError) as e:
        dfl.dflash_draft_block(h, a, L, rk, rv, 8, ws, topk=17)
    assert e.value.code == -2


def test_weights_beyond_fp16_range_are_rejected_at_create():
    dims = synth.DIMS["small"]
    W = synth.weights(dims, 95)
    W["layers"][1]["w_down"][3, 7] = 1.0e5                    # bf16 holds it, fp16 does not
    with pytest.raises(dfl.DflashError) as e:
        dfl.dflash_create(tu.lib_cfg(dims, batch_max=1, gamma_max=4), tu.to_dev(W))
    assert e.value.code == -9


def test_activation_beyond_fp16_range_is_reported():
    dims = synth.DIMS["small"]
    W = synth.weights(dims, 96)
    W["layers"][0]["g_mlp"] = W["layers"][0]["g_mlp"] * 1.0e5   # normed values ~N(0, 1e10)
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=1, gamma_max=4), tu.to_dev(W))
    rk, rv = synth.ring(dims, 1, 97)
    dev = torch.device("cuda")
    ws = dfl.workspace(dfl.dflash_draft_workspace_bytes(h))
    dfl.dflash_draft_block(h, torch.tensor([3], dtype=torch.int32, device=dev),
                           torch.tensor([50], dtype=torch.int64, device=dev), rk.cuda(), rv.cuda(), 4,
                           ws, out=dict(draft=torch.empty((1, 3), dtype=torch.int32, device=dev)))
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == -9


@pytest.mark.parametrize("gamma", [4, 16])
def test_ring_key_beyond_fp16_range_is_reported(gamma):
    """Attention reads ring keys as fp16: a bf16 key beyond +-65504 written
    into the ring by the caller is not saturated silently — it becomes
    infinite and the pass reports DFLASH_ERR_RANGE at its next fp16 store
    (gamma 4 and 16: 20 and 80 query rows per KV head)."""
    dims = synth.DIMS["small"]
    W = synth.weights(dims, 98)
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=1, gamma_max=16), tu.to_dev(W))
    rk, rv = synth.ring(dims, 1, 99)
    dev = torch.device("cuda")
    out = dict(draft=torch.empty((1, gamma - 1), dtype=torch.int32, device=dev))
    anchor = torch.tensor([3], dtype=torch.int32, device=dev)
    L = torch.tensor([200], dtype=torch.int64, device=dev)
    ws = dfl.workspace(dfl.dflash_draft_workspace_bytes(h))
    dfl.dflash_draft_block(h, anchor, L, rk.cuda(), rv.cuda(), gamma, ws, out=out)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    rk[1, 0, 1, 150, 17] = 1.0e5                 # layer 1, KV head 1, a visible slot
    ws2 = dfl.workspace(dfl.dflash_draft_workspace_bytes(h))
    dfl.dflash_draft_block(h, anchor, L, rk.cuda(), rv.cuda(), gamma, ws2, out=out)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws2) == -9

@pytest.mark.parametrize("gamma", [4, 16])
def test_masked_ring_slots_holding_nan_change_nothing(gamma):
    """Ring slots past the visible window that hold NaN in K and V change
    nothing: the pass matches the oracle, whose definition ignores those
    slots (it reads zeros there).  Context 200 of a 256-slot window: the last
    key tile is partly visible."""
    from oracle import model as om
    dims = synth.DIMS["small"]
    W = synth.weights(dims, 98)
    rk, rv = synth.ring(dims, 1, 99)
    L = torch.tensor([200], dtype=torch.int64)
    anchor = torch.tensor([3], dtype=torch.int32)
    ref = om.draft_pass(tu.oracle_cfg(dims), W, rk, rv, L.numpy(), anchor.numpy(), gamma)
    want = ref["logits"].reshape(1, gamma - 1, -1)
    rk_nan, rv_nan = rk.clone(), rv.clone()
    rk_nan[:, 0, :, 200:, :] = float("nan")
    rv_nan[:, 0, :, 230:, :] = float("nan")
    h = dfl.dflash_create(tu.lib_cfg(dims, batch_max=1, gamma_max=16), tu.to_dev(W))
    got = tu.run_draft(h, anchor, L, rk_nan.cuda(), rv_nan.cuda(), gamma, topk=4)
    assert tu.rel_err(got["logits"], want) <= 1e-2
