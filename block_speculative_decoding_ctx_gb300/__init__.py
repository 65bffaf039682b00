"""GB300-native single-pass block drafting with target-context injection and
lossless verification.

This module is a thin ctypes binding over ``libdflash.so`` (built from
``csrc/`` by ``build.py``).  Every function carries the name of the C entry
point it calls and only marshals arguments: torch tensors supply device memory
and the current CUDA stream; all computation runs in the library's kernels.
There is no fallback: if the library is missing, every call raises.
"""

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdflash.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "dflash.h")

DFLASH_VERIFY_GREEDY = 0
DFLASH_VERIFY_SAMPLED = 1

ERRORS = {
    -1: "DFLASH_ERR_ARG", -2: "DFLASH_ERR_SHAPE", -3: "DFLASH_ERR_ALIGN",
    -4: "DFLASH_ERR_UNSUPPORTED", -5: "DFLASH_ERR_LAUNCH", -6: "DFLASH_ERR_DEVICE_TIMEOUT",
    -7: "DFLASH_ERR_WORKSPACE", -8: "DFLASH_ERR_CUDA", -9: "DFLASH_ERR_RANGE",
}


class DflashError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        self.name = ERRORS.get(code, str(code))
        super().__init__(f"{where}: {self.name} ({dflash_strerror(code)})")


class dflash_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "n_layers", "n_feat",
        "feat_dim", "window", "gamma_max", "topk_max", "batch_max", "append_max")] + [
        ("rope_theta", ctypes.c_float), ("eps", ctypes.c_float), ("mask_id", ctypes.c_int),
        ("weight_format", ctypes.c_int)]


DFLASH_WEIGHTS_BF16 = 0
DFLASH_WEIGHTS_E4M3 = 1

LAYER_MATRICES = ("w_qkv", "w_o", "w_gate", "w_up", "w_down")


class dflash_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "g_attn", "w_qkv", "w_o", "g_mlp", "w_gate", "w_up", "w_down",
        "s_qkv", "s_o", "s_gate", "s_up", "s_down")]


class dflash_weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("lm_head", ctypes.c_void_p), ("w_c", ctypes.c_void_p),
                ("g_c", ctypes.c_void_p), ("g_final", ctypes.c_void_p),
                ("layers", ctypes.POINTER(dflash_layer_weights)), ("s_lm_head", ctypes.c_void_p)]


class dflash_sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_p", ctypes.c_float),
                ("seeds", ctypes.c_void_p), ("step", ctypes.c_uint64)]


class dflash_draft_out(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "topk_ids", "topk_vals", "lse", "logits", "q", "draft")]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


def lib():
    """Load libdflash.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "block_speculative_decoding_ctx_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    sig = {
        "dflash_create": (_I, [ctypes.POINTER(dflash_config), ctypes.POINTER(dflash_weights),
                               ctypes.POINTER(_P)]),
        "dflash_destroy": (_I, [_P]),
        "dflash_draft_workspace_bytes": (_SZ, [_P]),
        "dflash_append_workspace_bytes": (_SZ, [_P]),
        "dflash_verify_workspace_bytes": (_SZ, [_I, _I, _I]),
        "dflash_probs_workspace_bytes": (_SZ, [_I, _I]),
        "dflash_ctx_append": (_I, [_P, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P, _SZ, _P]),
        "dflash_draft_block": (_I, [_P, _I, _I, _P, _P, _P, _P, _P, _I, _I,
                                    ctypes.POINTER(dflash_sampling),
                                    ctypes.POINTER(dflash_draft_out), _P, _SZ, _P]),
        "dflash_probs": (_I, [_I, _I, _P, ctypes.c_float, ctypes.c_float, _P, _P, _SZ, _P]),
        "dflash_verify": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, ctypes.c_uint64, _P, _P, _P, _P, _P,
                               _SZ, _P]),
        "dflash_read_status": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
        "dflash_strerror": (ctypes.c_char_p, [_I]),
        "dflash_selftest_timeout": (_I, [_P, ctypes.c_longlong, _P]),
        "dflash_sample_draft": (_I, [_I, _I, _I, _P, _P, ctypes.c_uint64, _P, _P, _SZ, _P]),
        "dflash_sample_workspace_bytes": (_SZ, [_I, _I]),
        "dflash_profile_enable": (_I, [_P, _I]),
        "dflash_quantize_e4m3": (_I, [_P, _I, _I, _P, _P, _P]),
        "dflash_verify_noalloc": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, ctypes.c_uint64, _P, _P, _P,
                                       _P, _P]),
        "dflash_profile_read": (_I, [_P, ctypes.POINTER(ctypes.c_float),
                                     ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I), _I,
                                     ctypes.POINTER(_I)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def declared_functions():
    """Names of the functions include/dflash.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_\w+)\s*\(", text)))


# ----------------------------------------------------------------- helpers

def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(code, where):
    if code != 0:
        raise DflashError(code, where)


def dflash_strerror(code):
    return lib().dflash_strerror(int(code)).decode()


def workspace(nbytes, device="cuda"):
    """A zero-filled, 256-byte-aligned workspace tensor of nbytes bytes."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------ entry points

class Handle:
    """Owns a dflash_handle and keeps the weight tensors alive."""

    def __init__(self, ptr, keep, cfg):
        self.ptr = ptr
        self._keep = keep
        self.cfg = cfg

    def __del__(self):
        try:
            if self.ptr:
                lib().dflash_destroy(self.ptr)
                self.ptr = None
        except Exception:
            pass


def dflash_create(cfg, weights):
    """cfg: dict with the dflash_config fields (weight_format defaults to
    DFLASH_WEIGHTS_BF16); weights: dict of CUDA tensors (matrices bf16, gains
    float32) with keys embed, lm_head, w_c, g_c, g_final and layers =
    [dict(g_attn, w_qkv, w_o, g_mlp, w_gate, w_up, w_down)].  With
    DFLASH_WEIGHTS_E4M3 the layer matrices and lm_head are uint8 E4M3 codes
    and s_qkv, s_o, s_gate, s_up, s_down (per layer) and s_lm_head their
    float32 row scales."""
    cfg = dict(cfg)
    cfg.setdefault("weight_format", DFLASH_WEIGHTS_BF16)
    c = dflash_config(**{k: cfg[k] for k, _ in dflash_config._fields_})
    layers = (dflash_layer_weights * len(weights["layers"]))()
    for i, lw in enumerate(weights["layers"]):
        for k, _ in dflash_layer_weights._fields_:
            t = lw.get(k)
            setattr(layers[i], k, t.data_ptr() if t is not None else None)
    s_head = weights.get("s_lm_head")
    w = dflash_weights(weights["embed"].data_ptr(), weights["lm_head"].data_ptr(),
                       weights["w_c"].data_ptr(), weights["g_c"].data_ptr(),
                       weights["g_final"].data_ptr(), layers,
                       s_head.data_ptr() if s_head is not None else None)
    out = ctypes.c_void_p()
    _check(lib().dflash_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(out)), "dflash_create")
    return Handle(out, (weights, layers), dict(cfg))


def dflash_destroy(handle):
    if handle.ptr:
        _check(lib().dflash_destroy(handle.ptr), "dflash_destroy")
        handle.ptr = None


def dflash_draft_workspace_bytes(handle):
    return int(lib().dflash_draft_workspace_bytes(handle.ptr))


def dflash_append_workspace_bytes(handle):
    return int(lib().dflash_append_workspace_bytes(handle.ptr))


def dflash_verify_workspace_bytes(batch, gamma, vocab):
    return int(lib().dflash_verify_workspace_bytes(batch, gamma, vocab))


def dflash_probs_workspace_bytes(rows, vocab):
    return int(lib().dflash_probs_workspace_bytes(rows, vocab))


def dflash_ctx_append(handle, feats, n_new, ctx_len, ring_k, ring_v, ws, req_slot=None,
                      stream=None):
    """feats bf16 [B, n_max, nf, fd]; n_new int32 [B]; ctx_len int64 [B] (in/out)."""
    B, n_max = feats.shape[0], feats.shape[1]
    _check(lib().dflash_ctx_append(handle.ptr, B, n_max, _ptr(feats), _ptr(n_new), _ptr(ctx_len),
                                   _ptr(req_slot), _ptr(ring_k), _ptr(ring_v), ring_k.shape[1],
                                   _ptr(ws), ws.numel(), _stream(stream)), "dflash_ctx_append")


def dflash_draft_block(handle, anchor, ctx_len, ring_k, ring_v, gamma, ws, topk=0, out=None,
                       sampling=None, req_slot=None, stream=None):
    """out: dict with any of topk_ids, topk_vals, lse, logits, q, draft (CUDA tensors).
    sampling: dict(temperature, top_p, seeds (uint64 as int64 tensor), step) or None."""
    out = out or {}
    o = dflash_draft_out(*[out[k].data_ptr() if out.get(k) is not None else None
                           for k, _ in dflash_draft_out._fields_])
    sp = None
    if sampling is not None:
        sp = ctypes.byref(dflash_sampling(float(sampling["temperature"]), float(sampling["top_p"]),
                                          sampling["seeds"].data_ptr(), int(sampling["step"])))
    _check(lib().dflash_draft_block(handle.ptr, anchor.shape[0], gamma, _ptr(anchor), _ptr(ctx_len),
                                    _ptr(req_slot), _ptr(ring_k), _ptr(ring_v), ring_k.shape[1],
                                    topk, sp, ctypes.byref(o), _ptr(ws), ws.numel(),
                                    _stream(stream)), "dflash_draft_block")


def dflash_probs(logits, temperature, top_p, probs, ws, stream=None):
    rows = logits.numel() // logits.shape[-1]
    _check(lib().dflash_probs(rows, logits.shape[-1], _ptr(logits), float(temperature),
                              float(top_p), _ptr(probs), _ptr(ws), ws.numel(), _stream(stream)),
           "dflash_probs")


def dflash_verify(mode, target, draft, accept_len, tokens, ws, q=None, seeds=None, step=0,
                  next_anchor=None, n_append=None, stream=None):
    """target: greedy target logits or sampled p, float32 [B, gamma, V]."""
    B, gamma, V = target.shape
    _check(lib().dflash_verify(int(mode), B, gamma, V, _ptr(target), _ptr(q), _ptr(draft),
                               _ptr(seeds), ctypes.c_uint64(int(step) & (2 ** 64 - 1)),
                               _ptr(accept_len), _ptr(tokens), _ptr(next_anchor), _ptr(n_append),
                               _ptr(ws), ws.numel(), _stream(stream)), "dflash_verify")


def dflash_read_status(ws, stream=None):
    v = ctypes.c_int32(0)
    _check(lib().dflash_read_status(_ptr(ws), ctypes.byref(v), _stream(stream)),
           "dflash_read_status")
    return v.value


def dflash_selftest_timeout(ws, limit_ns=1_000_000, stream=None):
    _check(lib().dflash_selftest_timeout(_ptr(ws), int(limit_ns), _stream(stream)),
           "dflash_selftest_timeout")


def dflash_sample_workspace_bytes(rows, vocab):
    return int(lib().dflash_sample_workspace_bytes(rows, vocab))


def dflash_sample_draft(q, seeds, step, y, ws, stream=None):
    """q float32 [B, G, V]; seeds uint64 (as int64) [B]; y int32 [B, G] out."""
    B, G, V = q.shape
    _check(lib().dflash_sample_draft(B, G, V, _ptr(q), _ptr(seeds), ctypes.c_uint64(int(step) & (2 ** 64 - 1)),
                                     _ptr(y), _ptr(ws), ws.numel(), _stream(stream)),
           "dflash_sample_draft")


def dflash_profile_enable(handle, n_pairs):
    _check(lib().dflash_profile_enable(handle.ptr, int(n_pairs)), "dflash_profile_enable")


PROFILE_KINDS = {0: "gemm", 1: "attention", 2: "norm", 3: "topk", 4: "sampling"}


def dflash_profile_read(handle, cap=128):
    """Per-launch (ms, algorithmic bytes, kind) of the last draft_block call."""
    ms = (ctypes.c_float * cap)()
    by = (ctypes.c_double * cap)()
    kd = (ctypes.c_int * cap)()
    n = ctypes.c_int(0)
    _check(lib().dflash_profile_read(handle.ptr, ms, by, kd, cap, ctypes.byref(n)),
           "dflash_profile_read")
    return [(ms[i], by[i], PROFILE_KINDS.get(kd[i], str(kd[i]))) for i in range(n.value)]


def dflash_verify_noalloc(mode, target, draft, accept_len, tokens, q=None, seeds=None, step=0,
                          next_anchor=None, n_append=None, stream=None):
    """dflash_verify without a workspace, for callers that cannot provide
    device memory: the scratch is a fixed array inside the library (see
    include/dflash.h for its size limit and for why overlapping calls race)."""
    B, gamma, V = target.shape
    _check(lib().dflash_verify_noalloc(int(mode), B, gamma, V, _ptr(target), _ptr(q), _ptr(draft),
                                       _ptr(seeds), ctypes.c_uint64(int(step) & (2 ** 64 - 1)),
                                       _ptr(accept_len), _ptr(tokens), _ptr(next_anchor),
                                       _ptr(n_append), _stream(stream)), "dflash_verify_noalloc")


def dflash_quantize_e4m3(w, codes, scales, stream=None):
    """w bf16 [rows, cols] -> codes uint8 [rows, cols], scales float32 [rows]."""
    rows, cols = w.shape
    _check(lib().dflash_quantize_e4m3(_ptr(w), rows, cols, _ptr(codes), _ptr(scales), _stream(stream)),
           "dflash_quantize_e4m3")


def quantize_weights_e4m3(weights, stream=None):
    """A copy of a bf16 weight dict (see dflash_create) whose layer matrices
    and lm_head are E4M3 codes with their row scales, made on the device by
    dflash_quantize_e4m3; embed, w_c and the gains are shared."""
    def q(t):
        codes = torch.empty(t.shape, dtype=torch.uint8, device=t.device)
        scales = torch.empty(t.shape[0], dtype=torch.float32, device=t.device)
        dflash_quantize_e4m3(t, codes, scales, stream)
        return codes, scales

    out = {k: v for k, v in weights.items() if k != "layers"}
    out["lm_head"], out["s_lm_head"] = q(weights["lm_head"])
    out["layers"] = []
    for lw in weights["layers"]:
        nl = dict(lw)
        for k in LAYER_MATRICES:
            nl[k], nl["s_" + k[2:]] = q(lw[k])
        out["layers"].append(nl)
    return out
