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


def test_noalloc_verify_rejects_sizes_beyond_its_scratch():
    dfl.lib()
    dev = torch.device("cuda")
    B, gamma, V = 4096, 8, 16                 # tickets + argmax keys exceed 256 KiB
    tgt = torch.empty((B, gamma, V), device=dev)
    n, tok, _, _ = _outs(B, gamma)
    with pytest.raises(dfl.DflashError) as e:
        dfl.dflash_verify_noalloc(dfl.DFLASH_VERIFY_GREEDY, tgt, torch.zeros((B, gamma - 1), dtype=torch.int32,
                                                                             device=dev), n, tok)
    assert e.value.code == -2
