"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers in the shapes and distributions of the
workloads; it holds none of the method's arithmetic.  Every draw goes through
a seeded ``torch.Generator`` so that the same seed gives the same tensors in
the GPU path and in the CPU checker.

Workloads (dimensions of the drafter described by the model card
"Beam-1.0-501B-A23B-DFlash2", section "Model"; block sizes from the product
doc "Speculative decoding", section "How it works"):

  tiny    1 layer, hidden 256, 4 q / 2 KV heads of dim 64, SwiGLU 512,
          vocab 1,024, 5 feature layers of width 256, window 64, block 4;
  full    5 layers, hidden 5120, 40 q / 8 KV heads of dim 128, SwiGLU
          17,408, vocab 151,936, 5 feature layers of width 5120, window 4,096.

Weights are N(0, 0.02) rounded to bf16; RMSNorm gains are ones unless the
caller asks for random gains (tests do, so that a dropped gain is visible).
"""

import math

import torch

DIMS = {
    "tiny": dict(d=256, n_q=4, n_kv=2, hd=64, ffn=512, vocab=1024, n_layers=1,
                 n_feat=5, feat_dim=256, window=64),
    "full": dict(d=5120, n_q=40, n_kv=8, hd=128, ffn=17408, vocab=151936, n_layers=5,
                 n_feat=5, feat_dim=5120, window=4096),
    # several tiles in every dimension with a ragged vocabulary tail; query
    # group of 5 like the full model
    "small": dict(d=640, n_q=10, n_kv=2, hd=64, ffn=1408, vocab=5003, n_layers=2,
                  n_feat=5, feat_dim=384, window=256),
    # head dim 128 like the full model, ragged vocabulary
    "small128": dict(d=1280, n_q=10, n_kv=2, hd=128, ffn=2560, vocab=3001, n_layers=1,
                     n_feat=5, feat_dim=640, window=512),
    # enough weight tiles (SwiGLU 9728 = 152 x 64, vocabulary 20000) that batches
    # of 16-32 blocks take the persistent GEMM path
    "wide": dict(d=640, n_q=10, n_kv=2, hd=64, ffn=9728, vocab=20000, n_layers=1,
                 n_feat=5, feat_dim=384, window=256),
}


def gen(seed):
    return torch.Generator().manual_seed(int(seed))


def normal(shape, std, seed, dtype=torch.float32):
    t = torch.randn(shape, generator=gen(seed), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def weights(dims, seed, random_gains=False, std=0.02):
    """Drafter weights as CPU tensors: matrices bf16, gains float32."""
    d, hd = dims["d"], dims["hd"]
    qkv_rows = (dims["n_q"] + 2 * dims["n_kv"]) * hd
    s = int(seed) * 1000

    def gain(k):
        if random_gains:
            return 1.0 + normal((d,), 0.1, s + k)
        return torch.ones(d, dtype=torch.float32)

    W = {
        "embed": normal((dims["vocab"], d), std, s + 1, torch.bfloat16),
        "lm_head": normal((dims["vocab"], d), std, s + 2, torch.bfloat16),
        "w_c": normal((d, dims["n_feat"] * dims["feat_dim"]), std, s + 3, torch.bfloat16),
        "g_c": gain(4),
        "g_final": gain(5),
        "layers": [],
    }
    for l in range(dims["n_layers"]):
        b = s + 100 * (l + 1)
        W["layers"].append({
            "g_attn": gain(100 * (l + 1) + 8),
            "w_qkv": normal((qkv_rows, d), std, b + 2, torch.bfloat16),
            "w_o": normal((d, dims["n_q"] * hd), std, b + 3, torch.bfloat16),
            "g_mlp": gain(100 * (l + 1) + 9),
            "w_gate": normal((dims["ffn"], d), std, b + 5, torch.bfloat16),
            "w_up": normal((dims["ffn"], d), std, b + 6, torch.bfloat16),
            "w_down": normal((d, dims["ffn"]), std, b + 7, torch.bfloat16),
        })
    return W


def ring(dims, B, seed, std=1.0):
    """Context K/V ring caches [NL, B, Hkv, W, hd] bf16 filled with N(0, std)."""
    shape = (dims["n_layers"], B, dims["n_kv"], dims["window"], dims["hd"])
    return (normal(shape, std, seed * 7 + 1, torch.bfloat16),
            normal(shape, std, seed * 7 + 2, torch.bfloat16))


def features(dims, n, seed, dtype=torch.bfloat16):
    """Target hidden states of the five read layers [n, nf, fd], N(0, 1)."""
    return normal((n, dims["n_feat"], dims["feat_dim"]), 1.0, seed, dtype)


def token_ids(n, vocab, seed, exclude=None):
    g = gen(seed)
    ids = torch.randint(0, vocab, (n,), generator=g, dtype=torch.int64)
    if exclude is not None:
        ids = torch.where(ids == exclude, (ids + 1) % vocab, ids)
    return ids.to(torch.int32)


def log_uniform_lengths(n, lo, hi, seed):
    """Context lengths round(exp(U(ln lo, ln hi)))."""
    u = torch.rand(n, generator=gen(seed), dtype=torch.float64)
    return torch.round(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).to(torch.int64)


def seeds(n, seed):
    g = gen(seed)
    lo = torch.randint(0, 2 ** 31, (n,), generator=g, dtype=torch.int64)
    hi = torch.randint(0, 2 ** 31, (n,), generator=g, dtype=torch.int64)
    return (hi << 32) | lo
