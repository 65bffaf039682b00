"""GPU parity of the E4M3 (FP8) drafter weights.

The pages serve their models in FP8 without fixing a scheme; the library's
reading (E4M3, one float32 scale per output row, weights only) is written
out by the oracle (oracle/quant.py).  Here:

* dflash_quantize_e4m3 against the oracle's quantization, bit for bit
  (codes and scales);
* draft_block and ctx_append on a handle created from the device's own
  E4M3 weights against the oracle's pass over its own quantization of the
  same bf16 weights, dequantized exactly: logits within 1e-2 normwise, top-k
  tolerance-aware, log-sum-exp;
* dflash_create refuses NaN codes and scales that are not finite and
  positive."""

import numpy as np
import pytest
import torch

import block_speculative_decoding_ctx_gb300 as dfl
import dflash_testutil as tu
from block_speculative_decoding_ctx_gb300 import synth
from oracle import model as om
from oracle import quant

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dfl.lib()


def _quantize_on_device(w):
    codes = torch.empty(w.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(w.shape[0], dtype=torch.float32, device="cuda")
    dfl.dflash_quantize_e4m3(w.cuda(), codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("rows,cols,std", [(7, 64, 0.02), (300, 1408, 1.0), (129, 5120, 30.0)])
def test_quantize_matches_oracle_bit_exact(rows, cols, std):
    w = synth.normal((rows, cols), std, 500 + rows, torch.bfloat16)
    w[1] = 0.0                                       # a row of zeros: scale 1
    w[2, 5] = 1.0e4                                  # one large weight dominates its row
    # a row of exact ties once divided by its scale: 448 and (1 + 1/16) * 2^k
    w[3] = 0.0
    w[3, 0] = 448.0
    w[3, 1:9] = torch.tensor([1.0625, 1.1875, -1.0625, 2.125, 0.5, 3 * 2.0 ** -10, 2.0 ** -10, -2.0 ** -11])
    codes, scales = _quantize_on_device(w)
    want_codes, want_scales = quant.quantize_rows(w.float().numpy())
    np.testing.assert_array_equal(scales.view(np.uint32), want_scales.view(np.uint32))
    np.testing.assert_array_equal(codes, want_codes)


CASES = [
    # name, B, gamma, contexts: token tiles of 16, 32, 64 and 128 (two of them
    # at batch 32), a ragged vocabulary tail, head dims 64 and 128
    ("tiny", 2, 4, [64, 30]),
    ("small", 3, 8, [300, 17, 0]),
    ("small128", 2, 16, [512, 700]),
    ("small", 4, 8, [300, 17, 256, 1000]),
    ("wide", 8, 8, [300] * 4 + [17, 256, 0, 1000]),
    ("wide", 16, 8, [256] * 15 + [3]),
    ("wide", 32, 8, [300] * 31 + [40]),
]


@pytest.mark.parametrize("name,B,gamma,lens", CASES)
def test_e4m3_draft_block_matches_oracle(name, B, gamma, lens):
    dims = synth.DIMS[name]
    W = synth.weights(dims, 61, random_gains=True)
    W64, (ref_codes, ref_scales) = tu.oracle_e4m3_weights(W)
    Wq = dfl.quantize_weights_e4m3(tu.to_dev(W))
    np.testing.assert_array_equal(Wq["layers"][0]["w_qkv"].cpu().numpy(), ref_codes)
    np.testing.assert_array_equal(Wq["layers"][0]["s_qkv"].cpu().numpy(), ref_scales)
    rk, rv = synth.ring(dims, B, 62)
    anchor = synth.token_ids(B, dims["vocab"], 63)
    L = torch.tensor(lens, dtype=torch.int64)
    cfg = dict(tu.lib_cfg(dims, batch_max=B, gamma_max=max(gamma, 8)), weight_format=dfl.DFLASH_WEIGHTS_E4M3)
    h = dfl.dflash_create(cfg, Wq)
    got = tu.run_draft(h, anchor, L, rk.cuda(), rv.cuda(), gamma, topk=4)
    ref = om.draft_pass(tu.oracle_cfg(dims), W64, rk.double().numpy(), rv.double().numpy(), L.numpy(),
                        anchor.numpy(), gamma)
    want = ref["logits"]
    assert tu.rel_err(got["logits"], want) <= TOL
    flat = want.reshape(-1, want.shape[-1])
    tu.check_topk(got["topk_ids"].reshape(-1, 4), got["topk_vals"].reshape(-1, 4), flat, TOL)
    assert np.abs(got["lse"].reshape(-1) - om.logsumexp(flat)).max() <= TOL * np.abs(flat).max()


@pytest.mark.parametrize("name,B,n_max,starts,n_new", [("small", 3, 40, [5, 250, 1000], [40, 17, 0]),
                                                       ("small128", 2, 20, [511, 3], [20, 1]),
                                                       ("small", 2, 8, [5, 250], [8, 3])])
def test_e4m3_ctx_append_matches_oracle(name, B, n_max, starts, n_new):
    dims = synth.DIMS[name]
    W = synth.weights(dims, 64, random_gains=True)
    W64, _ = tu.oracle_e4m3_weights(W)
    feats = synth.features(dims, B * n_max, 65).reshape(B, n_max, dims["n_feat"], dims["feat_dim"])
    cfg = tu.oracle_cfg(dims)
    shape = (dims["n_layers"], B, dims["n_kv"], dims["window"], dims["hd"])
    want_k, want_v = np.zeros(shape), np.zeros(shape)
    for b in range(B):
        if n_new[b]:
            om.ctx_append(cfg, W64, want_k, want_v, b, feats[b, :n_new[b]], int(starts[b]))
    lc = dict(tu.lib_cfg(dims, batch_max=B, gamma_max=8, append_max=n_max),
              weight_format=dfl.DFLASH_WEIGHTS_E4M3)
    h = dfl.dflash_create(lc, dfl.quantize_weights_e4m3(tu.to_dev(W)))
    rk = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    rv = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    ctx = torch.tensor(starts, dtype=torch.int64, device="cuda")
    ws = dfl.workspace(dfl.dflash_append_workspace_bytes(h))
    dfl.dflash_ctx_append(h, feats.cuda(), torch.tensor(n_new, dtype=torch.int32, device="cuda"), ctx, rk, rv, ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    assert ctx.cpu().tolist() == [s + n for s, n in zip(starts, n_new)]
    assert tu.rel_err(rk.double().cpu().numpy(), want_k) <= TOL
    assert tu.rel_err(rv.double().cpu().numpy(), want_v) <= TOL


def test_e4m3_full_dims_batch1_matches_oracle():
    """The launch configuration of the benchmark's E4M3 line: full
    dimensions, batch 1, gamma 8, context 4,096, top-4."""
    dims = synth.DIMS["full"]
    W = synth.weights(dims, 66)
    W64, _ = tu.oracle_e4m3_weights(W)
    Wq = dfl.quantize_weights_e4m3(tu.to_dev(W))
    B, gamma = 1, 8
    rk, rv = synth.ring(dims, B, 67, std=1.4)
    anchor = synth.token_ids(B, dims["vocab"], 68)
    L = torch.tensor([4096], dtype=torch.int64)
    cfg = dict(tu.lib_cfg(dims, batch_max=B, gamma_max=gamma), weight_format=dfl.DFLASH_WEIGHTS_E4M3)
    h = dfl.dflash_create(cfg, Wq)
    got = tu.run_draft(h, anchor, L, rk.cuda(), rv.cuda(), gamma, topk=4)
    ref = om.draft_pass(tu.oracle_cfg(dims), W64, rk.double().numpy(), rv.double().numpy(), L.numpy(),
                        anchor.numpy(), gamma)
    want = ref["logits"]
    assert tu.rel_err(got["logits"], want) <= TOL
    flat = want.reshape(-1, want.shape[-1])
    tu.check_topk(got["topk_ids"].reshape(-1, 4), got["topk_vals"].reshape(-1, 4), flat, TOL)


def test_e4m3_create_refuses_nan_codes_and_bad_scales():
    dims = synth.DIMS["small"]
    W = synth.weights(dims, 69)
    cfg = dict(tu.lib_cfg(dims, batch_max=1, gamma_max=4), weight_format=dfl.DFLASH_WEIGHTS_E4M3)
    Wq = dfl.quantize_weights_e4m3(tu.to_dev(W))
    dfl.dflash_create(cfg, Wq)                                  # the good weights are accepted
    bad = dfl.quantize_weights_e4m3(tu.to_dev(W))
    bad["layers"][1]["w_down"][7, 3] = 0x7F                     # a NaN code
    with pytest.raises(dfl.DflashError) as e:
        dfl.dflash_create(cfg, bad)
    assert e.value.code == -9
    bad = dfl.quantize_weights_e4m3(tu.to_dev(W))
    bad["s_lm_head"][11] = float("inf")
    with pytest.raises(dfl.DflashError) as e:
        dfl.dflash_create(cfg, bad)
    assert e.value.code == -9
    bad = dfl.quantize_weights_e4m3(tu.to_dev(W))
    del bad["layers"][0]["s_o"]
    with pytest.raises(dfl.DflashError) as e:
        dfl.dflash_create(cfg, bad)
    assert e.value.code == -1
