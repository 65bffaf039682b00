"""Host-side checks of the C ABI: the library loads, exports every function
include/dflash.h declares, and rejects bad arguments before launching
anything (these calls never reach the GPU)."""

import ctypes

import pytest

import block_speculative_decoding_ctx_gb300 as dfl
from block_speculative_decoding_ctx_gb300 import build as dbuild


@pytest.fixture(scope="module")
def L():
    dbuild.build()
    return dfl.lib()


def test_library_exports_every_declared_function(L):
    names = dfl.declared_functions()
    assert {"dflash_ctx_append", "dflash_draft_block", "dflash_verify", "dflash_create"} <= set(names)
    missing = [n for n in names if not hasattr(L, n)]
    assert missing == []


def test_strerror_names_every_code(L):
    for code in dfl.ERRORS:
        assert dfl.dflash_strerror(code) != "unknown error code"
    assert dfl.dflash_strerror(0) == "ok"


def test_verify_rejects_bad_arguments_on_the_host(L):
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: validation fails first
    # bad mode
    assert L.dflash_verify(7, 1, 8, 100, fake, fake, fake, fake, 0, fake, fake, None, None, fake, 1 << 20, None) == -1
    # gamma < 2, vocab too large
    assert L.dflash_verify(0, 1, 1, 100, fake, None, fake, None, 0, fake, fake, None, None, fake, 1 << 20, None) == -2
    assert L.dflash_verify(0, 1, 8, 1 << 19, fake, None, fake, None, 0, fake, fake, None, None, fake, 1 << 20, None) == -2
    # null target / sampled without q
    assert L.dflash_verify(0, 1, 8, 100, None, None, fake, None, 0, fake, fake, None, None, fake, 1 << 20, None) == -1
    assert L.dflash_verify(1, 1, 8, 100, fake, None, fake, fake, 0, fake, fake, None, None, fake, 1 << 20, None) == -1
    # misaligned pointer
    assert L.dflash_verify(0, 1, 8, 100, P(4098), None, fake, None, 0, fake, fake, None, None, fake, 1 << 20, None) == -3
    # workspace too small
    need = dfl.dflash_verify_workspace_bytes(4, 8, 151936)
    assert need > 256
    assert L.dflash_verify(0, 4, 8, 151936, fake, None, fake, None, 0, fake, fake, None, None, fake, need - 1, None) == -7


def test_probs_rejects_bad_arguments_on_the_host(L):
    P = ctypes.c_void_p
    fake = P(4096)
    assert L.dflash_probs(4, 100, fake, 0.0, 0.9, P(8192), fake, 4096, None) == -1
    assert L.dflash_probs(4, 100, fake, 0.7, 1.5, P(8192), fake, 4096, None) == -1
    assert L.dflash_probs(4, 100, fake, 0.7, 0.9, fake, fake, 4096, None) == -1      # aliasing
    assert L.dflash_probs(0, 100, fake, 0.7, 0.9, P(8192), fake, 4096, None) == -2


def _cfg(**kw):
    c = dict(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=512, vocab=1024, n_layers=1,
             n_feat=5, feat_dim=256, window=64, gamma_max=8, topk_max=4, batch_max=4,
             append_max=64, rope_theta=1e6, eps=1e-6, mask_id=-1)
    c.update(kw)
    return dfl.dflash_config(**c)


def test_create_validates_the_configuration(L):
    lw = (dfl.dflash_layer_weights * 1)()
    for k, _ in dfl.dflash_layer_weights._fields_:
        setattr(lw[0], k, 4096)
    w = dfl.dflash_weights(4096, 4096, 4096, 4096, 4096, lw)
    out = ctypes.c_void_p()
    for bad, code in ((dict(head_dim=96), -4), (dict(n_q_heads=3), -2), (dict(gamma_max=17), -4),
                      (dict(hidden=200), -4), (dict(mask_id=5000), -1), (dict(topk_max=0), -4)):
        assert L.dflash_create(ctypes.byref(_cfg(**bad)), ctypes.byref(w), ctypes.byref(out)) == code
        assert not out.value
    # query rows of one KV head (group x gamma_max) are the rows of the attention MMAs: 144 > 128
    assert L.dflash_create(ctypes.byref(_cfg(n_q_heads=18, gamma_max=16)), ctypes.byref(w),
                           ctypes.byref(out)) == -4
    lw[0].w_o = 4100                       # misaligned weight
    assert L.dflash_create(ctypes.byref(_cfg()), ctypes.byref(w), ctypes.byref(out)) == -3
    # 128 rows pass the shape checks (the call then stops at the misaligned weight)
    assert L.dflash_create(ctypes.byref(_cfg(n_q_heads=16, gamma_max=16)), ctypes.byref(w),
                           ctypes.byref(out)) == -3
