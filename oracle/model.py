"""The block drafter, written out as plain float64 loops and library matmuls.

Test infrastructure only (see the package docstring).

Sources
  [blog]  "DFlash vs DFlash 2", sections "DFlash: generate the block all at
          once" (one masked, bidirectional pass over [anchor, MASK, ...];
          five Qwen-style layers; shared embedding and LM head) and
          "Conditioning on the target model" (H_t equation; Q/K/V injection
          equations; non-causal in-block attention).
  [card]  "Beam-1.0-501B-A23B-DFlash2" model card, section "Model" (5 layers,
          hidden 5120, 40 query / 8 KV heads of dim 128, SwiGLU 17,408,
          vocabulary 151,936, 4,096-token sliding window).
  [doc]   "Speculative decoding" product doc, section "How it works" (top
          candidates kept per position; window keeps draft cost flat).

Readings taken here where the pages are silent (parity with the oracle is
parity with these readings):
  * positions: RoPE (rotate-half pairs (j, j + hd/2), inv_freq_j =
    theta^(-2j/hd)) on queries and keys at absolute positions; context keys
    are rotated when appended; the block occupies positions L .. L+gamma-1
    where L is the number of context positions that have target features;
  * layer: pre-norm, x += Attn(RMSNorm(x)), x += MLP(RMSNorm(x)), then a final
    RMSNorm before the LM head; context K/V = W^K H_t, W^V H_t exactly as the
    injection equation writes them (no extra per-layer norm);
  * RMSNorm(x) = x / sqrt(mean(x^2) + eps) * g;
  * SwiGLU MLP: W_down (silu(W_gate h) * (W_up h));
  * attention: scale 1/sqrt(hd); one softmax over [context window ; block];
    context key at position s is visible iff L - W <= s < L; every block key
    is visible to every block query (non-causal); query head h reads KV head
    h // (Hq / Hkv);
  * output alignment: block row j >= 1 predicts x_{t+j}, so the LM head runs
    on the gamma - 1 MASK rows;
  * MASK is a token id (default V - 1) whose embedding row is looked up.

Layouts (row-major, torch Linear convention [out, in]):
  embed, lm_head [V, d]; w_c [d, nf*fd]; g_c [d];
  per layer: g_attn [d], w_qkv [(Hq + 2 Hkv) hd, d] (q rows, k rows, v rows),
  w_o [d, Hq hd], g_mlp [d], w_gate [F, d], w_up [F, d], w_down [d, F];
  g_final [d].
  Ring caches ring_k / ring_v [NL, B, Hkv, W, hd]; slot of position s = s mod W.
"""

from dataclasses import dataclass

import numpy as np


@dataclass
class Config:
    d: int
    n_q: int
    n_kv: int
    hd: int
    ffn: int
    vocab: int
    n_layers: int
    n_feat: int
    feat_dim: int
    window: int
    rope_theta: float = 1.0e6
    eps: float = 1.0e-6
    mask_id: int = -1            # -1 means vocab - 1

    @property
    def mask_token(self):
        return self.vocab - 1 if self.mask_id < 0 else self.mask_id


def weight_shapes(cfg):
    """Shapes of every drafter-owned matrix and gain (embed / LM head are shared)."""
    per_layer = {
        "g_attn": (cfg.d,),
        "w_qkv": ((cfg.n_q + 2 * cfg.n_kv) * cfg.hd, cfg.d),
        "w_o": (cfg.d, cfg.n_q * cfg.hd),
        "g_mlp": (cfg.d,),
        "w_gate": (cfg.ffn, cfg.d),
        "w_up": (cfg.ffn, cfg.d),
        "w_down": (cfg.d, cfg.ffn),
    }
    return {
        "w_c": (cfg.d, cfg.n_feat * cfg.feat_dim),
        "g_c": (cfg.d,),
        "layer": per_layer,
        "g_final": (cfg.d,),
    }


def drafter_matrix_params(cfg):
    """Parameter count of the drafter-owned matrices (layers + W_c)."""
    s = weight_shapes(cfg)
    per_layer = sum(int(np.prod(v)) for v in s["layer"].values() if len(v) == 2)
    return cfg.n_layers * per_layer + int(np.prod(s["w_c"]))


# ---------------------------------------------------------------- primitives

def f64(a):
    """Widen an array (numpy, or a torch CPU tensor of any float dtype)."""
    if hasattr(a, "detach"):
        a = a.detach().float().numpy()
    return np.asarray(a, dtype=np.float64)


def linear(x, w, chunk=16384):
    """y = x @ w.T with w [out, in]; w is widened in row chunks."""
    x = np.asarray(x, dtype=np.float64)
    out = w.shape[0]
    y = np.empty(x.shape[:-1] + (out,), dtype=np.float64)
    for r0 in range(0, out, chunk):
        r1 = min(out, r0 + chunk)
        y[..., r0:r1] = x @ f64(w[r0:r1]).T
    return y


def rmsnorm(x, g, eps):
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * f64(g)


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def rope(x, pos, theta):
    """Rotate-half RoPE.  x [..., n, hd]; pos broadcastable to x.shape[:-2]."""
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = np.asarray(pos, dtype=np.float64)[..., None, None] * inv_freq  # [..., 1, half]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ------------------------------------------------- target-feature injection

def fuse_features(cfg, W, feats):
    """H_t = RMSNorm(W_c [H^(l1); ... ; H^(l5)]).  feats [n, nf, fd] -> [n, d]."""
    f = f64(feats)
    n = f.shape[0]
    cat = f.reshape(n, cfg.n_feat * cfg.feat_dim)
    return rmsnorm(linear(cat, W["w_c"]), W["g_c"], cfg.eps)


def context_kv(cfg, W, H_t, positions):
    """Per layer i: K_i = RoPE(W^K_i H_t, pos), V_i = W^V_i H_t.

    Returns lists (one entry per layer) of [n, Hkv, hd] arrays.
    """
    qd = cfg.n_q * cfg.hd
    kd = cfg.n_kv * cfg.hd
    n = H_t.shape[0]
    Ks, Vs = [], []
    for lw in W["layers"]:
        k = linear(H_t, lw["w_qkv"][qd:qd + kd]).reshape(n, cfg.n_kv, cfg.hd)
        v = linear(H_t, lw["w_qkv"][qd + kd:qd + 2 * kd]).reshape(n, cfg.n_kv, cfg.hd)
        Ks.append(rope(k, np.asarray(positions), cfg.rope_theta))
        Vs.append(v)
    return Ks, Vs


def ctx_append(cfg, W, ring_k, ring_v, b, feats, start_pos):
    """Append positions start_pos .. start_pos+n-1 of request b to its ring.

    ring_k / ring_v: float64 [NL, B, Hkv, W, hd], updated in place.
    Returns H_t [n, d].
    """
    n = feats.shape[0]
    positions = start_pos + np.arange(n)
    H_t = fuse_features(cfg, W, feats)
    Ks, Vs = context_kv(cfg, W, H_t, positions)
    slots = positions % cfg.window
    for l in range(cfg.n_layers):
        for j in range(n):
            ring_k[l, b, :, slots[j], :] = Ks[l][j]
            ring_v[l, b, :, slots[j], :] = Vs[l][j]
    return H_t


# ---------------------------------------------------------- block attention

def slot_positions(L, W):
    """Absolute position held by each ring slot when positions < L were
    appended in order: the largest s < L with s = j (mod W), or -1."""
    j = np.arange(W)
    s = (L - 1) - np.mod(L - 1 - j, W)
    return np.where(s >= 0, s, -1)


def block_attention(cfg, q, k_blk, v_blk, ring_k_l, ring_v_l, L):
    """Brute-force attention of the block queries over [context ; block].

    q [G, Hq, hd]; k_blk, v_blk [G, Hkv, hd]; ring_*_l [Hkv, W, hd] (one
    request, one layer); L = context length.  Returns [G, Hq, hd].
    """
    G = q.shape[0]
    Wn = cfg.window
    s_pos = slot_positions(L, Wn)
    ctx_visible = (s_pos >= 0) & (s_pos >= L - Wn) & (s_pos < L)
    mask = np.concatenate([np.where(ctx_visible, 0.0, -np.inf),
                           np.zeros(G)])                       # [W + G]
    group = cfg.n_q // cfg.n_kv
    out = np.zeros((G, cfg.n_q, cfg.hd))
    scale = 1.0 / np.sqrt(cfg.hd)
    for h in range(cfg.n_q):
        g = h // group
        keys = np.concatenate([f64(ring_k_l[g]), k_blk[:, g, :]], axis=0)   # [W+G, hd]
        vals = np.concatenate([f64(ring_v_l[g]), v_blk[:, g, :]], axis=0)
        s = q[:, h, :] @ keys.T * scale + mask[None, :]                    # [G, W+G]
        s = s - s.max(axis=1, keepdims=True)
        pr = np.exp(s)
        pr = pr / pr.sum(axis=1, keepdims=True)
        out[:, h, :] = pr @ vals
    return out


# ------------------------------------------------------------ draft pass

def draft_pass(cfg, W, ring_k, ring_v, L, anchor, gamma, requests=None):
    """One single-pass block draft for each request.

    ring_k / ring_v [NL, B, Hkv, W, hd] (any float type); L [B] context
    lengths; anchor [B] token ids.  `requests` optionally restricts the pass to
    a subset of request indices.  Returns a dict with
      logits [b, gamma-1, V], final_hidden [b, gamma, d] (after the final
      RMSNorm), and layer_out: list of residual streams [b, gamma, d].
    """
    L = np.asarray(L)
    anchor = np.asarray(anchor)
    reqs = list(range(len(L))) if requests is None else list(requests)
    nb = len(reqs)
    ids = np.full((nb, gamma), cfg.mask_token, dtype=np.int64)
    ids[:, 0] = anchor[reqs]
    emb = W["embed"]
    x = np.stack([np.stack([f64(emb[int(t)]) for t in row]) for row in ids])  # [nb, gamma, d]
    pos = np.asarray([L[b] + np.arange(gamma) for b in reqs])                 # [nb, gamma]
    qd, kd = cfg.n_q * cfg.hd, cfg.n_kv * cfg.hd
    layer_out = []
    for l, lw in enumerate(W["layers"]):
        h = rmsnorm(x, lw["g_attn"], cfg.eps)
        qkv = linear(h, lw["w_qkv"])
        q = rope(qkv[..., :qd].reshape(nb, gamma, cfg.n_q, cfg.hd), pos, cfg.rope_theta)
        k = rope(qkv[..., qd:qd + kd].reshape(nb, gamma, cfg.n_kv, cfg.hd), pos, cfg.rope_theta)
        v = qkv[..., qd + kd:].reshape(nb, gamma, cfg.n_kv, cfg.hd)
        o = np.stack([block_attention(cfg, q[i], k[i], v[i], ring_k[l, b], ring_v[l, b], int(L[b]))
                      for i, b in enumerate(reqs)])
        x = x + linear(o.reshape(nb, gamma, qd), lw["w_o"])
        h = rmsnorm(x, lw["g_mlp"], cfg.eps)
        x = x + linear(silu(linear(h, lw["w_gate"])) * linear(h, lw["w_up"]), lw["w_down"])
        layer_out.append(x.copy())
    hf = rmsnorm(x, W["g_final"], cfg.eps)
    logits = linear(hf[:, 1:, :], W["lm_head"])
    return {"logits": logits, "final_hidden": hf, "layer_out": layer_out}


def topk(logits, k):
    """Top-k of each row: (ids, values), values descending, ties to lower id."""
    z = np.asarray(logits, dtype=np.float64)
    V = z.shape[-1]
    flat = z.reshape(-1, V)
    ids = np.empty((flat.shape[0], k), dtype=np.int64)
    for r in range(flat.shape[0]):
        order = np.lexsort((np.arange(V), -flat[r]))
        ids[r] = order[:k]
    ids = ids.reshape(z.shape[:-1] + (k,))
    vals = np.take_along_axis(z, ids, axis=-1)
    return ids, vals


def logsumexp(logits):
    z = np.asarray(logits, dtype=np.float64)
    m = z.max(axis=-1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))[..., 0]
