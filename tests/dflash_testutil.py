"""Helpers shared by the GPU parity tests (marshalling and comparisons)."""

import numpy as np
import torch

import block_speculative_decoding_ctx_gb300 as dfl
from oracle import model as om


def lib_cfg(dims, batch_max, gamma_max, topk_max=4, append_max=64, mask_id=-1):
    return dict(hidden=dims["d"], n_q_heads=dims["n_q"], n_kv_heads=dims["n_kv"], head_dim=dims["hd"],
                ffn=dims["ffn"], vocab=dims["vocab"], n_layers=dims["n_layers"],
                n_feat=dims["n_feat"], feat_dim=dims["feat_dim"], window=dims["window"],
                gamma_max=gamma_max, topk_max=topk_max, batch_max=batch_max,
                append_max=append_max, rope_theta=1.0e6, eps=1.0e-6, mask_id=mask_id)


def oracle_cfg(dims, mask_id=-1):
    return om.Config(**dims, mask_id=mask_id)


def to_dev(W, dev="cuda"):
    if isinstance(W, dict):
        return {k: to_dev(v, dev) for k, v in W.items()}
    if isinstance(W, list):
        return [to_dev(v, dev) for v in W]
    return W.to(dev).contiguous()


def rel_err(got, want):
    """max |got - want| / max |want| (normwise relative error)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.abs(got - want).max() / max(np.abs(want).max(), 1e-30))


def check_topk(ids, vals, logits_ref, tol):
    """Every GPU id's oracle logit reaches the oracle's k-th value within
    tol * max|logit|; ids are distinct; GPU values match the oracle logits of
    those ids within the same tolerance."""
    R, k = ids.shape
    scale = np.abs(logits_ref).max()
    for r in range(R):
        row = logits_ref[r]
        kth = np.sort(row)[::-1][k - 1]
        assert len(set(ids[r].tolist())) == k
        assert (row[ids[r]] >= kth - tol * scale).all()
        assert np.abs(vals[r] - row[ids[r]]).max() <= tol * scale
        assert (np.diff(vals[r]) <= 0).all()


def run_draft(h, anchor, ctx_len, rk, rv, gamma, topk, sampling=None, req_slot=None, with_logits=True):
    dev = torch.device("cuda")
    B = anchor.shape[0]
    V = h.cfg["vocab"]
    R = B * (gamma - 1)
    out = dict(topk_ids=torch.full((B, gamma - 1, max(topk, 1)), -7, dtype=torch.int32, device=dev)
               if topk else None,
               topk_vals=torch.full((B, gamma - 1, max(topk, 1)), -7.0, device=dev) if topk else None,
               lse=torch.full((B, gamma - 1), -7.0, device=dev),
               logits=torch.full((B, gamma - 1, V), -7.0, device=dev) if with_logits else None,
               q=torch.full((B, gamma - 1, V), -7.0, device=dev) if sampling else None,
               draft=torch.full((B, gamma - 1), -7, dtype=torch.int32, device=dev))
    ws = dfl.workspace(dfl.dflash_draft_workspace_bytes(h))
    dfl.dflash_draft_block(h, anchor.to(dev), ctx_len.to(dev), rk, rv, gamma, ws, topk=topk, out=out,
                           sampling=sampling, req_slot=req_slot)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    assert R > 0
    return {k: (v.cpu().numpy() if v is not None else None) for k, v in out.items()}


def widen(W):
    """Float64 numpy copies of CPU weight tensors (exact: bf16 and float32
    values are float64 values).  The oracle reads them without re-widening
    per call, which keeps full-size oracle passes to seconds."""
    if isinstance(W, dict):
        return {k: widen(v) for k, v in W.items()}
    if isinstance(W, list):
        return [widen(v) for v in W]
    return W.double().numpy()


def check_probs(got, want, tol=1e-5):
    """A float32 sampling distribution against the oracle's float64 one, row
    by row: the kept sets may differ only in a few ids at the nucleus boundary
    whose mass is below tol; on the ids both keep, max abs error over max abs
    value <= tol."""
    got = got.reshape(-1, got.shape[-1])
    want = want.reshape(-1, want.shape[-1])
    np.testing.assert_allclose(got.sum(-1), 1.0, rtol=1e-4)
    for r in range(got.shape[0]):
        kg, kw = got[r] > 0, want[r] > 0
        diff = kg ^ kw
        assert want[r][diff].sum() <= tol and diff.sum() <= 3
        both = kg & kw
        assert np.abs(got[r][both] - want[r][both]).max() / np.abs(want[r]).max() <= tol


def check_q_against_oracle_logits(q_gpu, z_gpu, z_ref, T, top_p):
    """q = top_p(softmax(z / T)) from the drafter's logits, judged through the
    logits it came from.

    With eps = max |z_gpu - z_ref| over a row, every log-probability of
    softmax(z / T) moves by at most 2 eps / T (eps / T for the id itself, as
    much again for the log-sum-exp), and renormalising a nucleus that keeps
    the same ids moves it by at most as much again: 4 eps / T in all.  So,
    per row and per id kept on both sides,
        |q_gpu - q_ref| <= (exp(4 eps / T) - 1) * max(q_gpu, q_ref),
    and an id kept on one side only lies at the nucleus boundary: it is no
    more likely than exp(4 eps / T) times the least likely id both keep.
    Returns the largest eps seen (the logits themselves are checked by the
    caller against the 1e-2 normwise bar)."""
    from oracle import sampling as osamp
    V = q_gpu.shape[-1]
    qg = q_gpu.reshape(-1, V).astype(np.float64)
    zg = z_gpu.reshape(-1, V).astype(np.float64)
    zr = z_ref.reshape(-1, V)
    worst = 0.0
    for r in range(qg.shape[0]):
        eps = float(np.abs(zg[r] - zr[r]).max())
        worst = max(worst, eps)
        qr = osamp.probs(zr[r:r + 1], T, top_p)[0]
        f = np.exp(4.0 * eps / T)
        kg, kr = qg[r] > 0, qr > 0
        both = kg & kr
        assert (np.abs(qg[r][both] - qr[both]) <= (f - 1.0) * np.maximum(qg[r][both], qr[both]) + 1e-12).all()
        floor = min(qg[r][both].min(), qr[both].min())
        assert (qg[r][kg & ~kr] <= f * floor).all() and (qr[kr & ~kg] <= f * floor).all()
    return worst


def oracle_e4m3_weights(W, chunk_rows=1024):
    """Float64 weights the oracle reads for an E4M3 drafter: every layer
    matrix and the LM head quantized by the oracle's own E4M3 rule from the
    same bf16 values and dequantized exactly (code value times row scale);
    embed, w_c and the gains widened as they are.  Also returns the oracle's
    codes and scales of layer 0's w_qkv for a bit-exact check."""
    from oracle import quant

    import concurrent.futures
    import os

    def deq(t):
        out = np.empty(t.shape, dtype=np.float64)

        def one(r0):
            codes, s = quant.quantize_rows(t[r0:r0 + chunk_rows].float().numpy())
            out[r0:r0 + chunk_rows] = quant.dequantize_rows(codes, s)

        # rows are independent; numpy releases the interpreter lock in its loops
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
            list(ex.map(one, range(0, t.shape[0], chunk_rows)))
        return out

    W64 = {k: (widen(v) if k != "layers" else None) for k, v in W.items()}
    W64["lm_head"] = deq(W["lm_head"])
    W64["layers"] = []
    for lw in W["layers"]:
        d = {k: widen(v) for k, v in lw.items()}
        for k in ("w_qkv", "w_o", "w_gate", "w_up", "w_down"):
            d[k] = deq(lw[k])
        W64["layers"].append(d)
    ref_codes = quant.quantize_rows(W["layers"][0]["w_qkv"].float().numpy())
    return W64, ref_codes
