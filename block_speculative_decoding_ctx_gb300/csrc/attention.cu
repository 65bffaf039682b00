// Launcher of the drafter's block attention: the gamma block queries of every
// query head attend over [context window ; whole block], non-causally inside
// the block ("DFlash vs DFlash 2" blog, section "Conditioning on the target
// model": K_i = [W^K H_t ; W^K H_d], V_i = [W^V H_t ; W^V H_d]; block
// positions attend to one another non-causally; model card
// "Beam-1.0-501B-A23B-DFlash2", section "Model": 4,096-token sliding window,
// 40 query / 8 KV heads).  The kernel is attn_tc_kernel (attention_tc.cu);
// here the ring's tensor maps are encoded and the shape is checked.
#include "attention.h"
#include "common.cuh"
#include "gemm.h"

namespace dfl {
namespace {

constexpr int kKeys = 64;  // keys per ring tile: the height of the TMA box

}  // namespace

int attn_max_rows() { return 128; }

int launch_attention(const void* ring_k_layer, const void* ring_v_layer, const AttnArgs& a, int B,
                     cudaStream_t s) {
  if (!attention_tc_supported(a)) return DFLASH_ERR_UNSUPPORTED;
  CUtensorMap tk, tv;
  const uint64_t rows = (uint64_t)a.ring_batch * a.n_kv * a.window;
  int rc = encode_2d(&tk, ring_k_layer, OPND_BF16, (uint64_t)a.hd, rows, 64, kKeys);
  if (rc) return rc;
  rc = encode_2d(&tv, ring_v_layer, OPND_BF16, (uint64_t)a.hd, rows, 64, kKeys);
  if (rc) return rc;
  return launch_attention_tc(tk, tv, a, B, s);
}

}  // namespace dfl
