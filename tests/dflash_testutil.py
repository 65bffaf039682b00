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


def run_draft(h, anchor, ctx_len, rk, rv, gamma, topk, sampling=None, req_slot=None):
    dev = torch.device("cuda")
    B = anchor.shape[0]
    V = h.cfg["vocab"]
    R = B * (gamma - 1)
    out = dict(topk_ids=torch.full((B, gamma - 1, max(topk, 1)), -7, dtype=torch.int32, device=dev)
               if topk else None,
               topk_vals=torch.full((B, gamma - 1, max(topk, 1)), -7.0, device=dev) if topk else None,
               lse=torch.full((B, gamma - 1), -7.0, device=dev),
               logits=torch.full((B, gamma - 1, V), -7.0, device=dev),
               q=torch.full((B, gamma - 1, V), -7.0, device=dev) if sampling else None,
               draft=torch.full((B, gamma - 1), -7, dtype=torch.int32, device=dev))
    ws = dfl.workspace(dfl.dflash_draft_workspace_bytes(h))
    dfl.dflash_draft_block(h, anchor.to(dev), ctx_len.to(dev), rk, rv, gamma, ws, topk=topk, out=out,
                           sampling=sampling, req_slot=req_slot)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    assert R > 0
    return {k: (v.cpu().numpy() if v is not None else None) for k, v in out.items()}
