// C ABI: handle, context injection and the single-pass block draft.
// See include/dflash.h for the contract of every entry point.
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "kernels.h"

using namespace dfl;

struct dflash_handle {
  dflash_config cfg;
  dflash_weights w;
  std::vector<dflash_layer_weights> layers;
};

namespace {

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) % 16) == 0; }

int validate_config(const dflash_config& c) {
  if (c.hidden < 64 || c.hidden % 64) return DFLASH_ERR_UNSUPPORTED;
  if (c.head_dim != 64 && c.head_dim != 128) return DFLASH_ERR_UNSUPPORTED;
  if (c.n_q_heads < 1 || c.n_kv_heads < 1 || c.n_q_heads % c.n_kv_heads) return DFLASH_ERR_SHAPE;
  if ((c.n_q_heads * c.head_dim) % 64) return DFLASH_ERR_UNSUPPORTED;
  if (c.ffn < 64 || c.ffn % 64) return DFLASH_ERR_UNSUPPORTED;
  if (c.vocab < 2 || c.vocab > (1 << 18)) return DFLASH_ERR_SHAPE;
  if (c.n_layers < 1 || c.n_layers > 64) return DFLASH_ERR_SHAPE;
  if (c.n_feat < 1 || c.feat_dim < 1 || (c.n_feat * c.feat_dim) % 64) return DFLASH_ERR_UNSUPPORTED;
  if (c.window < 1) return DFLASH_ERR_SHAPE;
  if (c.gamma_max < 2 || c.gamma_max > 16) return DFLASH_ERR_UNSUPPORTED;
  if (c.topk_max < 1 || c.topk_max > 16) return DFLASH_ERR_UNSUPPORTED;
  if (c.batch_max < 1 || c.batch_max > 256) return DFLASH_ERR_UNSUPPORTED;
  if (c.append_max < 1 || c.append_max > 8192) return DFLASH_ERR_UNSUPPORTED;
  if (!(c.eps > 0.0f) || !(c.rope_theta > 0.0f)) return DFLASH_ERR_ARG;
  if (c.mask_id < -1 || c.mask_id >= c.vocab) return DFLASH_ERR_ARG;
  return DFLASH_OK;
}

}  // namespace

extern "C" {

int dflash_create(const dflash_config* cfg, const dflash_weights* w, dflash_handle** out) {
  if (!out) return DFLASH_ERR_ARG;
  *out = nullptr;
  if (!cfg || !w || !w->layers) return DFLASH_ERR_ARG;
  int rc = validate_config(*cfg);
  if (rc) return rc;
  const void* top[] = {w->embed, w->lm_head, w->w_c, w->g_c, w->g_final};
  for (const void* p : top)
    if (!aligned16(p)) return p ? DFLASH_ERR_ALIGN : DFLASH_ERR_ARG;
  for (int l = 0; l < cfg->n_layers; ++l) {
    const dflash_layer_weights& L = w->layers[l];
    const void* ps[] = {L.g_attn, L.w_qkv, L.w_o, L.g_mlp, L.w_gate, L.w_up, L.w_down};
    for (const void* p : ps)
      if (!aligned16(p)) return p ? DFLASH_ERR_ALIGN : DFLASH_ERR_ARG;
  }
  dflash_handle* h = new (std::nothrow) dflash_handle;
  if (!h) return DFLASH_ERR_ARG;
  h->cfg = *cfg;
  h->w = *w;
  h->layers.assign(w->layers, w->layers + cfg->n_layers);
  h->w.layers = h->layers.data();
  *out = h;
  return DFLASH_OK;
}

int dflash_destroy(dflash_handle* h) {
  delete h;
  return DFLASH_OK;
}

size_t dflash_draft_workspace_bytes(const dflash_handle* h) { return h ? kWsHeader : 0; }
size_t dflash_append_workspace_bytes(const dflash_handle* h) { return h ? kWsHeader : 0; }

int dflash_ctx_append(dflash_handle* h, int B, int n_max, const void* feats, const int32_t* n_new,
                      int64_t* ctx_len, const int32_t* req_slot, void* ring_k, void* ring_v,
                      int ring_batch, void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  (void)h; (void)B; (void)n_max; (void)feats; (void)n_new; (void)ctx_len; (void)req_slot;
  (void)ring_k; (void)ring_v; (void)ring_batch; (void)workspace; (void)ws_bytes; (void)stream;
  return DFLASH_ERR_UNSUPPORTED;
}

int dflash_draft_block(dflash_handle* h, int B, int gamma, const int32_t* anchor,
                       const int64_t* ctx_len, const int32_t* req_slot, const void* ring_k,
                       const void* ring_v, int ring_batch, int topk, const dflash_sampling* sampling,
                       const dflash_draft_out* out, void* workspace, size_t ws_bytes,
                       dflash_stream_t stream) {
  (void)h; (void)B; (void)gamma; (void)anchor; (void)ctx_len; (void)req_slot; (void)ring_k;
  (void)ring_v; (void)ring_batch; (void)topk; (void)sampling; (void)out; (void)workspace;
  (void)ws_bytes; (void)stream;
  return DFLASH_ERR_UNSUPPORTED;
}

}  // extern "C"
