"""GPU parity of verification and sampling preparation against the oracle.

Accept lengths and committed tokens must be bit-exact given the same float32
p / q and the same Philox streams; sampling distributions must match the
oracle within 1e-5 (max abs error over max abs value, float32 vs float64).
Inputs follow the verify sweep recipe: draft logits N(0, 3), target logits =
draft logits + N(0, sigma), p and q their softmax."""

import numpy as np
import pytest
import torch

import block_speculative_decoding_ctx_gb300 as dfl
from block_speculative_decoding_ctx_gb300 import synth
from oracle import sampling as osamp
from oracle import verify as over

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dfl.lib()


def _probs_f32(logits):
    out = np.empty(logits.shape, dtype=np.float32)
    flat_in = logits.reshape(-1, logits.shape[-1])
    flat_out = out.reshape(-1, logits.shape[-1])
    for r0 in range(0, flat_in.shape[0], 64):
        flat_out[r0:r0 + 64] = osamp.probs(flat_in[r0:r0 + 64]).astype(np.float32)
    return out


def _sweep_inputs(B, gamma, V, sigma, seed):
    d = synth.normal((B, gamma, V), 3.0, seed).numpy()
    t = d + synth.normal((B, gamma, V), sigma, seed + 1).numpy()
    p = _probs_f32(t)
    q = _probs_f32(d[:, :gamma - 1])
    seeds = synth.seeds(B, seed + 2).numpy().view(np.uint64)
    y = osamp.draft_draw(q, seeds, 3).astype(np.int32)
    return t.astype(np.float32), p, q, y, seeds


def _run_verify(mode, target, draft, q=None, seeds=None, step=0):
    B, gamma, V = target.shape
    dev = torch.device("cuda")
    tt = torch.from_numpy(np.ascontiguousarray(target)).to(dev)
    dd = torch.from_numpy(np.ascontiguousarray(draft)).to(dev)
    qq = None if q is None else torch.from_numpy(np.ascontiguousarray(q)).to(dev)
    ss = None if seeds is None else torch.from_numpy(seeds.view(np.int64).copy()).to(dev)
    n = torch.full((B,), -7, dtype=torch.int32, device=dev)
    tok = torch.full((B, gamma), -7, dtype=torch.int32, device=dev)
    ws = dfl.workspace(dfl.dflash_verify_workspace_bytes(B, gamma, V))
    outs = []
    for _ in range(2):                      # second call checks the self-reset scratch
        dfl.dflash_verify(mode, tt, dd, n, tok, ws, q=qq, seeds=ss, step=step)
        torch.cuda.synchronize()
        outs.append((n.cpu().numpy().copy(), tok.cpu().numpy().copy()))
    assert dfl.dflash_read_status(ws) == 0
    assert (outs[0][0] == outs[1][0]).all() and (outs[0][1] == outs[1][1]).all()
    return outs[0]


@pytest.mark.parametrize("B,gamma,V", [(1, 4, 1024), (3, 8, 5003), (16, 8, 151936), (1, 16, 151936)])
def test_greedy_verify_bit_exact(B, gamma, V):
    rng = np.random.default_rng(B * 100 + gamma)
    t = synth.normal((B, gamma, V), 1.0, 11 + B).numpy()
    a = t.argmax(-1)
    y = np.empty((B, gamma - 1), dtype=np.int32)
    for b in range(B):
        k = int(rng.integers(0, gamma))            # accept exactly k drafts
        y[b] = a[b, :gamma - 1]
        if k < gamma - 1:
            y[b, k] = (a[b, k] + 1 + rng.integers(0, V - 1)) % V
    want_n, want_tok = over.greedy(t, y)
    got_n, got_tok = _run_verify(dfl.DFLASH_VERIFY_GREEDY, t, y)
    np.testing.assert_array_equal(got_n, want_n)
    np.testing.assert_array_equal(got_tok, want_tok)


def test_greedy_verify_ties_go_to_lowest_id():
    t = np.zeros((2, 4, 300), dtype=np.float32)
    t[:, :, 7] = 2.0
    t[:, :, 250] = 2.0                 # tie across chunks / threads
    t[1, 2, 100] = 2.0
    y = np.array([[7, 7, 7], [7, 7, 250]], dtype=np.int32)
    want = over.greedy(t, y)
    got = _run_verify(dfl.DFLASH_VERIFY_GREEDY, t, y)
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1], want[1])


@pytest.mark.parametrize("B,gamma,V,sigma", [(1, 4, 1024, 1.0), (7, 8, 5003, 0.25),
                                             (32, 16, 151936, 1.0), (256, 8, 151936, 4.0)])
def test_sampled_verify_bit_exact(B, gamma, V, sigma):
    _, p, q, y, seeds = _sweep_inputs(B, gamma, V, sigma, 1000 + B)
    want_n, want_tok = over.sampled(p, q, y, seeds, 3)
    got_n, got_tok = _run_verify(dfl.DFLASH_VERIFY_SAMPLED, p, y, q=q, seeds=seeds, step=3)
    np.testing.assert_array_equal(got_n, want_n)
    np.testing.assert_array_equal(got_tok, want_tok)
    assert 0 < want_n.mean() < gamma - 1 or B < 8


def test_sampled_verify_edge_cases():
    """p = q (always accept, bonus), one-hot q on an impossible token (always
    reject, residual = p), and a large step that uses the counter's high word."""
    B, gamma, V = 4, 5, 777
    rng = np.random.default_rng(5)
    p = rng.dirichlet(np.ones(V), size=(B, gamma)).astype(np.float32)
    q = p[:, :gamma - 1].copy()
    q[2:] = 0.0
    q[2:, :, 5] = 1.0
    p[2:, 0, 5] = 0.0
    seeds = np.array([1, 2, 3, 2 ** 63 + 5], dtype=np.uint64)
    y = osamp.draft_draw(q, seeds, 2 ** 40 + 9).astype(np.int32)
    want = over.sampled(p, q, y, seeds, 2 ** 40 + 9)
    got = _run_verify(dfl.DFLASH_VERIFY_SAMPLED, p, y, q=q, seeds=seeds, step=2 ** 40 + 9)
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1], want[1])
    assert (want[0][:2] == gamma - 1).all() and (want[0][2:] == 0).all()


def _run_probs(logits, T, top_p):
    dev = torch.device("cuda")
    lt = torch.from_numpy(logits).to(dev)
    out = torch.full_like(lt, -1.0)
    ws = dfl.workspace(dfl.dflash_probs_workspace_bytes(lt.shape[0], lt.shape[1]))
    dfl.dflash_probs(lt, T, top_p, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("rows,V,T,top_p", [(3, 1024, 1.0, 1.0), (5, 5003, 0.7, 0.99),
                                            (9, 151936, 0.7, 0.99), (4, 151936, 0.7, 0.5)])
def test_probs_matches_oracle(rows, V, T, top_p):
    logits = synth.normal((rows, V), 1.4, 77 + rows).numpy()
    got = _run_probs(logits, T, top_p)
    want = osamp.probs(logits, T, top_p)
    np.testing.assert_allclose(got.sum(-1), 1.0, rtol=1e-4)
    for r in range(rows):
        kg, kw = got[r] > 0, want[r] > 0
        diff = kg ^ kw                      # only ids at the nucleus boundary may differ
        assert want[r][diff].sum() <= 1e-5 and diff.sum() <= 3
        both = kg & kw
        err = np.abs(got[r][both] - want[r][both]).max() / np.abs(want[r]).max()
        assert err <= 1e-5


def test_probs_ties_keep_lowest_ids():
    """A nucleus boundary inside a group of equal probabilities keeps the
    lowest ids of the group."""
    V = 64
    logits = np.zeros((1, V), dtype=np.float32)
    logits[0, :4] = 3.0
    got = _run_probs(logits, 1.0, 0.95)
    want = osamp.probs(logits, 1.0, 0.95)
    np.testing.assert_array_equal(got > 0, want > 0)
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-7)


def test_bounded_wait_gives_up_and_context_stays_usable():
    ws = dfl.workspace(256)
    dfl.dflash_selftest_timeout(ws, 1_000_000)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == -6
    # the context still runs work
    test_greedy_verify_bit_exact(1, 4, 1024)
