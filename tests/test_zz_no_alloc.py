"""The allocation-free verify entry point, for callers that cannot provide
device memory when they verify (a serving process whose device memory is
reserved up front by another allocator, or a host framework that forbids
plug-ins from allocating): dflash_verify_noalloc keeps its scratch in a fixed
array inside the library.  Its results must equal those of dflash_verify
(which takes a caller workspace) bit for bit — accept lengths, committed
tokens and the commit outputs — on two calls in a row, since every call reuses
the same array.  This file is collected last on purpose."""

import numpy as np
import pytest
import torch

import block_speculative_decoding_ctx_gb300 as dfl
from block_speculative_decoding_ctx_gb300 import synth

pytestmark = pytest.mark.gpu


def _inputs(B, gamma, V, seed):
    g = torch.Generator().manual_seed(seed)
    d = torch.randn((B, gamma, V), generator=g) * 3.0
    t = d + torch.randn((B, gamma, V), generator=g)
    p = torch.softmax(t, dim=-1)
    q = torch.softmax(d[:, :gamma - 1], dim=-1)
    draft = torch.multinomial(q.reshape(-1, V), 1, generator=g).reshape(B, gamma - 1).to(torch.int32)
    seeds = synth.seeds(B, seed + 1)
    return t.float(), p.float(), q.float(), draft, seeds


def _outs(B, gamma):
    dev = torch.device("cuda")
    return (torch.full((B,), -9, dtype=torch.int32, device=dev),
            torch.full((B, gamma), -9, dtype=torch.int32, device=dev),
            torch.full((B,), -9, dtype=torch.int32, device=dev),
            torch.full((B,), -9, dtype=torch.int32, device=dev))


@pytest.mark.parametrize("mode", [dfl.DFLASH_VERIFY_GREEDY, dfl.DFLASH_VERIFY_SAMPLED])
@pytest.mark.parametrize("B,gamma,V", [(3, 8, 5003), (16, 8, 151936)])
def test_noalloc_verify_matches_workspace_verify_twice(mode, B, gamma, V):
    dfl.lib()
    dev = torch.device("cuda")
    t, p, q, draft, seeds = _inputs(B, gamma, V, 100 + B + mode)
    target = (t if mode == dfl.DFLASH_VERIFY_GREEDY else p).to(dev)
    qd = q.to(dev) if mode == dfl.DFLASH_VERIFY_SAMPLED else None
    sd = seeds.to(dev) if mode == dfl.DFLASH_VERIFY_SAMPLED else None
    dd = draft.to(dev)
    if mode == dfl.DFLASH_VERIFY_GREEDY:
        # make some drafts match the target's choice so accept lengths vary
        a = t.argmax(-1)[:, :gamma - 1].to(torch.int32)
        for b in range(B):
            k = b % gamma
            dd[b, :k] = a[b, :k].to(dev)
    ref = _outs(B, gamma)
    ws = dfl.workspace(dfl.dflash_verify_workspace_bytes(B, gamma, V))
    dfl.dflash_verify(mode, target, dd, ref[0], ref[1], ws, q=qd, seeds=sd, step=7,
                      next_anchor=ref[2], n_append=ref[3])
    torch.cuda.synchronize()
    for _ in range(2):
        got = _outs(B, gamma)
        dfl.dflash_verify_noalloc(mode, target, dd, got[0], got[1], q=qd, seeds=sd, step=7,
                                  next_anchor=got[2], n_append=got[3])
        torch.cuda.synchronize()
        for r, g_ in zip(ref, got):
            np.testing.assert_array_equal(g_.cpu().numpy(), r.cpu().numpy())


def _device_inputs(B, gamma, V, seed):
    """The same recipe drawn on the device (the boundary case holds ~6 GB per
    tensor)."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(seed)
    d = torch.randn((B, gamma, V), generator=g, device=dev) * 3.0
    t = d + torch.randn((B, gamma, V), generator=g, device=dev)
    p = torch.softmax(t, dim=-1)
    del t
    q = torch.softmax(d[:, :gamma - 1], dim=-1)
    del d
    draft = torch.multinomial(q.reshape(-1, V), 1, generator=g).reshape(B, gamma - 1).to(torch.int32)
    seeds = synth.seeds(B, seed + 1).to(dev)
    return p, q, draft, seeds


def test_noalloc_verify_at_its_largest_batch_and_one_beyond():
    """At gamma 16 and vocabulary 151,936 the scratch holds B = 600 (exactly
    256 KiB after rounding) and not B = 601: 600 matches dflash_verify, 601 is
    refused and leaves its outputs untouched."""
    dfl.lib()
    gamma, V = 16, 151936
    p, q, draft, seeds = _device_inputs(601, gamma, V, 600)
    B = 600
    ref = _outs(B, gamma)
    ws = dfl.workspace(dfl.dflash_verify_workspace_bytes(B, gamma, V))
    dfl.dflash_verify(dfl.DFLASH_VERIFY_SAMPLED, p[:B], draft[:B], ref[0], ref[1], ws, q=q[:B],
                      seeds=seeds[:B], step=9, next_anchor=ref[2], n_append=ref[3])
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    for _ in range(2):
        got = _outs(B, gamma)
        dfl.dflash_verify_noalloc(dfl.DFLASH_VERIFY_SAMPLED, p[:B], draft[:B], got[0], got[1], q=q[:B],
                                  seeds=seeds[:B], step=9, next_anchor=got[2], n_append=got[3])
        torch.cuda.synchronize()
        for r, g_ in zip(ref, got):
            np.testing.assert_array_equal(g_.cpu().numpy(), r.cpu().numpy())
    over = _outs(601, gamma)
    with pytest.raises(dfl.DflashError) as e:
        dfl.dflash_verify_noalloc(dfl.DFLASH_VERIFY_SAMPLED, p, draft, over[0], over[1], q=q, seeds=seeds,
                                  step=9, next_anchor=over[2], n_append=over[3])
    assert e.value.code == -2
    torch.cuda.synchronize()
    for o in over:
        assert (o == -9).all()


def test_noalloc_verify_rejects_sizes_beyond_its_scratch():
    dfl.lib()
    dev = torch.device("cuda")
    B, gamma, V = 4096, 8, 16                 # tickets + argmax keys exceed 256 KiB
    tgt = torch.empty((B, gamma, V), device=dev)
    n, tok, anc, app = _outs(B, gamma)
    with pytest.raises(dfl.DflashError) as e:
        dfl.dflash_verify_noalloc(dfl.DFLASH_VERIFY_GREEDY, tgt, torch.zeros((B, gamma - 1), dtype=torch.int32,
                                                                             device=dev), n, tok,
                                  next_anchor=anc, n_append=app)
    assert e.value.code == -2
    torch.cuda.synchronize()
    for o in (n, tok, anc, app):
        assert (o == -9).all()                # nothing was launched
