// C ABI: handle, context injection and the single-pass block draft.
// See include/dflash.h for the contract of every entry point.
//
// ctx_append  ("DFlash vs DFlash 2" blog, section "Conditioning on the target
//              model", H_t equation and K/V injection equation):
//   W_c GEMM (bf16 features) -> RMSNorm(g_c) (fp16) -> per-layer K/V GEMM
//   whose epilogue rotates K and scatters K and V into ring slot pos mod W ->
//   ctx_len += n; up to 32 tokens the RMSNorm is folded into the two GEMMs.
// draft_block ("DFlash: generate the block all at once"):
//   embed [anchor, MASK...] + RMSNorm (+RoPE table) -> for each layer: QKV
//   GEMM (+RoPE) -> block attention over [ring window ; block] -> O GEMM ->
//   residual add + RMSNorm -> gate|up GEMM (+SwiGLU) -> down GEMM -> residual
//   add + RMSNorm (final RMSNorm gathers the gamma-1 MASK rows) -> LM head GEMM
//   (fp32 logits, then a chunked top-k + log-sum-exp kernel; or, when no
//   logits are wanted, an epilogue that keeps each vocabulary tile's top keys
//   and (max, sum of exp), then a merge kernel) [-> q = top_p(softmax(logits
//   / T)) -> y ~ q].
// Every drafter contraction runs on fp16 operands: the handle holds an fp16
// copy of the matrices (exact re-encoding of the bf16 values) and every
// activation between kernels is stored as fp16.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "attention.h"
#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "rowops.h"

using namespace dfl;

constexpr size_t kGemmPartialFloats = 4u << 20;  // ticketed split-K partial tiles (16 MiB)
constexpr int kGemmCounters = 8192;
constexpr int kFreeResidTokens = 64;

struct LayerMaps {
  CUtensorMap qkv, o, gate, up, down;  // over the fp16 copies
};

struct dflash_handle {
  dflash_config cfg;
  dflash_weights w;
  std::vector<dflash_layer_weights> layers;
  std::vector<LayerMaps> maps;
  CUtensorMap lm_head, w_c;  // lm_head: fp16 copy; w_c: the caller's bf16 matrix
  RopeInv rope;              // inverse rotary frequencies (double -> float pairs)
  void* f16 = nullptr;       // fp16 copies of every layer's matrices and the LM head (bf16 weights)
  int wtype = OPND_F16;      // operand type of those matrices in the GEMMs (OPND_E4M3: in place)
  int num_sms;
  int mask_id;
  // benchmark hook: device completion timestamps of draft_block's launches
  unsigned long long* prof_ts = nullptr;  // [prof_cap + 1], device
  int prof_cap = 0;
  std::vector<double> prof_bytes;
  std::vector<int> prof_kinds;
  int prof_used = 0;
};

namespace {


bool aligned(const void* p, size_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int validate_config(const dflash_config& c) {
  if (c.hidden < 64 || c.hidden % 64 || c.hidden > 12288) return DFLASH_ERR_UNSUPPORTED;
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
  if (c.weight_format != DFLASH_WEIGHTS_BF16 && c.weight_format != DFLASH_WEIGHTS_E4M3) return DFLASH_ERR_ARG;
  // query-group rows of one KV head are the rows of the attention MMAs
  if ((c.n_q_heads / c.n_kv_heads) * c.gamma_max > attn_max_rows()) return DFLASH_ERR_UNSUPPORTED;
  return DFLASH_OK;
}

// Key splits per (request, KV head): the largest power of two (<= 16; the
// attention launcher caps it to the largest cluster the GPU can co-schedule)
// that keeps B * Hkv * splits CTAs within one CTA per SM.  Splitting further
// was measured slower on GB300: at batch 16 two splits cost 16% over one,
// at batch 32 four splits 37% — the cluster merge costs more than the tail.
int attn_splits(const dflash_handle* h, int B) {
  const int bh = B * h->cfg.n_kv_heads;
  const int tiles = (h->cfg.window + 63) / 64;
  const int want = h->num_sms / bh > 1 ? h->num_sms / bh : 1;
  int s = 1;
  while (s * 2 <= want && s * 2 <= tiles && s * 2 <= 16) s *= 2;
  return s;
}

struct DraftWs {
  int* status;
  int* gemm_counters;
  int* topk_counters;
  int* samp_counters;
  float* x;
  float* y;
  void* h;
  void* qkv;
  void* attn;
  void* mlp;
  void* hf;
  float* logits;
  float2* rope_cs;
  float* ssq;  // [hidden / 128][M] per-tile sums of squares of the stream
  float* gemm_partial;
  unsigned long long* topk_keys;  // chunked top-k partials over the fp32 logits
  float* topk_ml;
  unsigned long long* tk_keys;  // LM-head epilogue top-k partials [R][vocab tiles][slots]
  float2* tk_ml;                // [R][vocab tiles]
  unsigned long long* samp_zsum;
  size_t bytes;
};

DraftWs draft_layout(const dflash_handle* h, void* base) {
  const dflash_config& c = h->cfg;
  const size_t M = (size_t)c.batch_max * c.gamma_max;
  const size_t R = (size_t)c.batch_max * (c.gamma_max - 1);
  const int qkv_dim = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  const int q_dim = c.n_q_heads * c.head_dim;
  const int chunks = row_chunks(c.vocab);
  Carve cv(base, kWsHeader);
  DraftWs w;
  w.status = static_cast<int*>(base);
  w.gemm_counters = cv.take<int>(kGemmCounters);
  w.topk_counters = cv.take<int>(R);
  w.samp_counters = cv.take<int>(R);
  // fp32 residual stream; fp16 GEMM operands
  w.x = cv.take<float>(M * c.hidden);
  w.y = cv.take<float>(M * c.hidden);  // O / down output before its residual add
  w.h = cv.take<uint16_t>(M * c.hidden);
  w.qkv = cv.take<uint16_t>(M * qkv_dim);
  w.attn = cv.take<uint16_t>(M * q_dim);
  w.mlp = cv.take<uint16_t>(M * c.ffn);
  w.hf = cv.take<uint16_t>(R * c.hidden);
  w.logits = cv.take<float>(R * c.vocab);
  w.rope_cs = cv.take<float2>(M * (c.head_dim / 2));
  w.ssq = cv.take<float>((size_t)((c.hidden + 127) / 128) * M);
  w.gemm_partial = cv.take<float>(kGemmPartialFloats);
  w.topk_keys = cv.take<unsigned long long>(R * chunks * 16);
  w.topk_ml = cv.take<float>(R * chunks * 2);
  const size_t vtiles = (size_t)((c.vocab + 127) / 128);
  w.tk_keys = cv.take<unsigned long long>(R * vtiles * topk_slots(c.topk_max));
  w.tk_ml = cv.take<float2>(R * vtiles);
  w.samp_zsum = cv.take<unsigned long long>(R * chunks);
  w.bytes = cv.off;
  return w;
}

struct AppendWs {
  int* status;
  int* gemm_counters;
  float* fused;
  float* gemm_partial;
  void* ht;
  float2* rope_cs;
  float* ssq;  // [hidden / 128][M] per-tile sums of squares of W_c's output (folded RMSNorm)
  size_t bytes;
};

AppendWs append_layout(const dflash_handle* h, void* base) {
  const dflash_config& c = h->cfg;
  const size_t M = (size_t)c.batch_max * c.append_max;
  Carve cv(base, kWsHeader);
  AppendWs w;
  w.status = static_cast<int*>(base);
  w.gemm_counters = cv.take<int>(kGemmCounters);
  w.fused = cv.take<float>(M * c.hidden);
  w.ht = cv.take<uint16_t>(M * c.hidden);
  w.rope_cs = cv.take<float2>(M * (c.head_dim / 2));
  w.ssq = cv.take<float>((size_t)((c.hidden + 127) / 128) * (M < 32 ? 32 : M));
  w.gemm_partial = cv.take<float>(kGemmPartialFloats);
  w.bytes = cv.off;
  return w;
}

GemmAOpts single_map(const float* scale = nullptr) {
  GemmAOpts o;
  o.n_maps = 1;
  o.tiles_per_map = 1 << 30;
  o.row_offset = 0;
  o.dual = 0;
  for (int i = 0; i < kMaxAMaps; ++i) o.scale[i] = nullptr;
  o.scale[0] = scale;
  return o;
}

GemmEpi epi_base(int kind, int M, int N, void* out, long long ld, int* status) {
  GemmEpi e;
  std::memset(&e, 0, sizeof(e));
  e.kind = kind;
  e.M = M;
  e.N = N;
  e.out = out;
  e.ld = ld;
  e.status = status;
  return e;
}

// inv_freq_j = theta^(-2j/hd) in double, kept as a float pair for the kernels.
RopeInv rope_inv(const dflash_config& c) {
  RopeInv r;
  const int half = c.head_dim / 2;
  for (int j = 0; j < 64; ++j) {
    const double inv = j < half ? std::pow((double)c.rope_theta, -2.0 * j / c.head_dim) : 0.0;
    const float hi = (float)inv;
    r.f[j] = make_float2(hi, (float)(inv - (double)hi));
  }
  return r;
}

int splits_for(const dflash_handle* h, int n_tiles, int M, int K) {
  const int BN = gemm_token_tile_for(M, n_tiles, h->num_sms);
  const int m_tiles = (M + BN - 1) / BN;
  const int per_sm = BN <= 64 ? 2 : 1;
  return gemm_plan_splits(n_tiles * m_tiles, K, h->num_sms * per_sm);
}

// Profiling marks (no-ops unless enabled).  A mark is a one-warp kernel
// launched with programmatic dependent launch right after a launch of the
// pass: it lets the next kernel be scheduled at once (so that kernel's early
// start overlaps the profiled one exactly as without the mark), waits for the
// profiled kernel to complete and writes %globaltimer into its slot.  Slot 0
// is written by a mark before the first launch.  Launch i is then charged the
// interval between completions i and i + 1: the intervals add up to the
// whole pass, overlap included, where an event pair around every launch
// would serialise neighbouring kernels and charge each its full latency.
__global__ void profile_mark_kernel(unsigned long long* ts, int slot) {
  pdl_enter();
  if (threadIdx.x == 0) ts[slot] = globaltimer_ns();
}

bool prof_mark(dflash_handle* h, cudaStream_t s, int slot) {
  return launch_pdl(profile_mark_kernel, dim3(1), dim3(32), 0, s, h->prof_ts, slot) == DFLASH_OK;
}
int prof_begin(dflash_handle* h, cudaStream_t s) {
  const int i = h->prof_used;
  if (i >= h->prof_cap) return -1;
  if (i == 0 && !prof_mark(h, s, 0)) return -1;
  return i;
}
void prof_end(dflash_handle* h, cudaStream_t s, int slot, double bytes, int kind) {
  if (slot < 0) return;
  if (!prof_mark(h, s, slot + 1)) return;
  h->prof_bytes[slot] = bytes;
  h->prof_kinds[slot] = kind;
  h->prof_used = slot + 1;
}

// Launch one draft GEMM.  bytes = algorithmic bytes of the launch.
int draft_gemm(dflash_handle* h, const GemmAMaps& A, const GemmAOpts& ao, int n_tiles, const void* x,
               int M, int K, const GemmEpi& e, const GemmScratch& sc, cudaStream_t s, double bytes,
               const GemmRowScale* rs = nullptr) {
  const int slot = prof_begin(h, s);
  const int rc = launch_gemm(A, ao, n_tiles, x, h->wtype, M, K, e, sc, splits_for(h, n_tiles, M, K),
                             s, true, rs);
  if (rc) return rc;
  prof_end(h, s, slot, bytes, DFLASH_KIND_GEMM);
  return DFLASH_OK;
}

// E4M3 weights: check the caller's codes and scales, then encode the TMA
// descriptors over them in place (no copy).
int create_e4m3(dflash_handle* h, const dflash_weights& w) {
  const dflash_config& c = h->cfg;
  const uint64_t d = c.hidden, F = c.ffn, qd = (uint64_t)c.n_q_heads * c.head_dim;
  const uint64_t qkv_rows = (uint64_t)(c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  h->wtype = OPND_E4M3;
  struct Mat {
    const void* codes;
    const float* scale;
    uint64_t rows, cols;
  };
  std::vector<Mat> mats;
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& L = h->layers[l];
    mats.push_back({L.w_qkv, L.s_qkv, qkv_rows, d});
    mats.push_back({L.w_o, L.s_o, d, qd});
    mats.push_back({L.w_gate, L.s_gate, F, d});
    mats.push_back({L.w_up, L.s_up, F, d});
    mats.push_back({L.w_down, L.s_down, d, F});
  }
  mats.push_back({w.lm_head, w.s_lm_head, (uint64_t)c.vocab, d});
  for (const Mat& m : mats) {
    if (!m.scale) return DFLASH_ERR_ARG;
    if (!aligned(m.scale, 4)) return DFLASH_ERR_ALIGN;
  }
  int* flag = nullptr;
  if (cudaMalloc(&flag, sizeof(int)) != cudaSuccess) {
    (void)cudaGetLastError();
    return DFLASH_ERR_CUDA;
  }
  // the weights may have been written on any stream: wait for all of it
  int rc = cudaDeviceSynchronize() == cudaSuccess && cudaMemset(flag, 0, sizeof(int)) == cudaSuccess
               ? DFLASH_OK
               : DFLASH_ERR_CUDA;
  for (size_t i = 0; i < mats.size() && !rc; ++i)
    rc = launch_check_e4m3(mats[i].codes, mats[i].rows * mats[i].cols, mats[i].scale, mats[i].rows, flag,
                           4 * h->num_sms, 0);
  int bad = 0;
  if (!rc && cudaMemcpy(&bad, flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) rc = DFLASH_ERR_CUDA;
  cudaFree(flag);
  if (rc) return rc;
  if (bad) return DFLASH_ERR_RANGE;
  h->maps.resize(c.n_layers);
  rc = encode_2d_u8(&h->lm_head, w.lm_head, d, c.vocab, 128, 128);
  if (!rc) rc = encode_2d(&h->w_c, w.w_c, OPND_BF16, (uint64_t)c.n_feat * c.feat_dim, d, 64, 128);
  for (int l = 0; l < c.n_layers && !rc; ++l) {
    const dflash_layer_weights& L = h->layers[l];
    LayerMaps& m = h->maps[l];
    rc = encode_2d_u8(&m.qkv, L.w_qkv, d, qkv_rows, 128, 128);
    if (!rc) rc = encode_2d_u8(&m.o, L.w_o, qd, d, 128, 128);
    if (!rc) rc = encode_2d_u8(&m.gate, L.w_gate, d, F, 128, 64);
    if (!rc) rc = encode_2d_u8(&m.up, L.w_up, d, F, 128, 64);
    if (!rc) rc = encode_2d_u8(&m.down, L.w_down, F, d, 128, 128);
  }
  return rc;
}

}  // namespace

extern "C" {

int dflash_quantize_e4m3(const void* w, int rows, int cols, void* codes, float* scales,
                         dflash_stream_t stream) {
  if (!w || !codes || !scales) return DFLASH_ERR_ARG;
  if (rows < 1 || cols < 16 || cols % 16) return DFLASH_ERR_SHAPE;
  if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return DFLASH_ERR_ALIGN;
  return launch_quantize_e4m3(w, rows, cols, codes, scales, reinterpret_cast<cudaStream_t>(stream));
}

int dflash_profile_enable(dflash_handle* h, int n_pairs) {
  if (!h || n_pairs < 0 || n_pairs > 4096) return DFLASH_ERR_ARG;
  if (h->prof_ts) cudaFree(h->prof_ts);
  h->prof_ts = nullptr;
  h->prof_cap = 0;
  h->prof_bytes.assign(n_pairs, 0.0);
  h->prof_kinds.assign(n_pairs, 0);
  h->prof_used = 0;
  if (n_pairs == 0) return DFLASH_OK;
  void* p = nullptr;
  if (cudaMalloc(&p, sizeof(unsigned long long) * (n_pairs + 1)) != cudaSuccess) {
    (void)cudaGetLastError();
    return DFLASH_ERR_CUDA;
  }
  h->prof_ts = static_cast<unsigned long long*>(p);
  h->prof_cap = n_pairs;
  return DFLASH_OK;
}

int dflash_profile_read(dflash_handle* h, float* ms, double* bytes, int* kinds, int cap, int* count) {
  if (!h || !count || cap < 0 || (cap > 0 && (!ms || !bytes || !kinds))) return DFLASH_ERR_ARG;
  const int n = h->prof_used < cap ? h->prof_used : cap;
  *count = 0;
  if (n == 0) return DFLASH_OK;
  std::vector<unsigned long long> ts(h->prof_used + 1);
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(ts.data(), h->prof_ts, sizeof(unsigned long long) * ts.size(),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  for (int i = 0; i < n; ++i) {
    ms[i] = (float)((double)(long long)(ts[i + 1] - ts[i]) * 1e-6);
    bytes[i] = h->prof_bytes[i];
    kinds[i] = h->prof_kinds[i];
  }
  *count = n;
  return DFLASH_OK;
}

int dflash_create(const dflash_config* cfg, const dflash_weights* w, dflash_handle** out) {
  if (!out) return DFLASH_ERR_ARG;
  *out = nullptr;
  if (!cfg || !w || !w->layers) return DFLASH_ERR_ARG;
  int rc = validate_config(*cfg);
  if (rc) return rc;
  const void* top[] = {w->embed, w->lm_head, w->w_c, w->g_c, w->g_final};
  for (const void* p : top)
    if (!aligned(p, 16)) return p ? DFLASH_ERR_ALIGN : DFLASH_ERR_ARG;
  for (int l = 0; l < cfg->n_layers; ++l) {
    const dflash_layer_weights& L = w->layers[l];
    const void* ps[] = {L.g_attn, L.w_qkv, L.w_o, L.g_mlp, L.w_gate, L.w_up, L.w_down};
    for (const void* p : ps)
      if (!aligned(p, 16)) return p ? DFLASH_ERR_ALIGN : DFLASH_ERR_ARG;
  }
  dflash_handle* h = new (std::nothrow) dflash_handle;
  if (!h) return DFLASH_ERR_ARG;
  h->cfg = *cfg;
  h->w = *w;
  h->layers.assign(w->layers, w->layers + cfg->n_layers);
  h->w.layers = h->layers.data();
  h->mask_id = cfg->mask_id < 0 ? cfg->vocab - 1 : cfg->mask_id;
  h->rope = rope_inv(*cfg);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    delete h;
    return DFLASH_ERR_CUDA;
  }
  const dflash_config& c = *cfg;
  const uint64_t d = c.hidden, F = c.ffn, qd = (uint64_t)c.n_q_heads * c.head_dim;
  const uint64_t qkv_rows = (uint64_t)(c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  if (c.weight_format == DFLASH_WEIGHTS_E4M3) {
    rc = create_e4m3(h, *w);
    if (rc) {
      dflash_destroy(h);
      return rc;
    }
    *out = h;
    return DFLASH_OK;
  }

  // fp16 copies: per layer qkv, o, gate, up, down, then the LM head; a flag word last
  struct Mat {
    const void* src;
    size_t n;
    size_t off;
  };
  std::vector<Mat> mats;
  size_t total = 0;
  auto add = [&](const void* src, size_t n) {
    mats.push_back({src, n, total});
    total += align_up(n * 2, 256);
  };
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& L = h->layers[l];
    add(L.w_qkv, qkv_rows * d);
    add(L.w_o, d * qd);
    add(L.w_gate, F * d);
    add(L.w_up, F * d);
    add(L.w_down, d * F);
  }
  add(w->lm_head, (size_t)c.vocab * d);
  if (cudaMalloc(&h->f16, total + 256) != cudaSuccess) {
    (void)cudaGetLastError();
    h->f16 = nullptr;
    dflash_destroy(h);
    return DFLASH_ERR_CUDA;
  }
  char* base = static_cast<char*>(h->f16);
  int* flag = reinterpret_cast<int*>(base + total);
  // the weights may have been written on any stream: wait for all of it
  rc = cudaDeviceSynchronize() == cudaSuccess && cudaMemset(flag, 0, sizeof(int)) == cudaSuccess
           ? DFLASH_OK
           : DFLASH_ERR_CUDA;
  for (size_t i = 0; i < mats.size() && !rc; ++i)
    rc = launch_to_f16(mats[i].src, base + mats[i].off, mats[i].n, flag, 4 * h->num_sms, 0);
  int bad = 0;
  if (!rc && cudaMemcpy(&bad, flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    rc = DFLASH_ERR_CUDA;
  if (!rc && bad) rc = DFLASH_ERR_RANGE;

  h->maps.resize(c.n_layers);
  auto mat = [&](size_t i) { return static_cast<const void*>(base + mats[i].off); };
  if (!rc) rc = encode_2d(&h->lm_head, mat(mats.size() - 1), OPND_F16, d, c.vocab, 64, 128);
  if (!rc) rc = encode_2d(&h->w_c, w->w_c, OPND_BF16, (uint64_t)c.n_feat * c.feat_dim, d, 64, 128);
  for (int l = 0; l < c.n_layers && !rc; ++l) {
    LayerMaps& m = h->maps[l];
    const size_t i = (size_t)l * 5;
    rc = encode_2d(&m.qkv, mat(i), OPND_F16, d, qkv_rows, 64, 128);
    if (!rc) rc = encode_2d(&m.o, mat(i + 1), OPND_F16, qd, d, 64, 128);
    if (!rc) rc = encode_2d(&m.gate, mat(i + 2), OPND_F16, d, F, 64, 64);
    if (!rc) rc = encode_2d(&m.up, mat(i + 3), OPND_F16, d, F, 64, 64);
    if (!rc) rc = encode_2d(&m.down, mat(i + 4), OPND_F16, F, d, 64, 128);
  }
  if (rc) {
    dflash_destroy(h);
    return rc;
  }
  *out = h;
  return DFLASH_OK;
}

int dflash_destroy(dflash_handle* h) {
  if (h) {
    if (h->prof_ts) cudaFree(h->prof_ts);
    if (h->f16) cudaFree(h->f16);
  }
  delete h;
  return DFLASH_OK;
}

size_t dflash_draft_workspace_bytes(const dflash_handle* h) {
  return h ? draft_layout(h, nullptr).bytes : 0;
}

size_t dflash_append_workspace_bytes(const dflash_handle* h) {
  return h ? append_layout(h, nullptr).bytes : 0;
}

int dflash_ctx_append(dflash_handle* h, int B, int n_max, const void* feats, const int32_t* n_new,
                      int64_t* ctx_len, const int32_t* req_slot, void* ring_k, void* ring_v,
                      int ring_batch, void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  if (!h) return DFLASH_ERR_ARG;
  const dflash_config& c = h->cfg;
  if (B < 1 || B > c.batch_max || n_max < 1 || n_max > c.append_max) return DFLASH_ERR_SHAPE;
  if (ring_batch < 1 || (!req_slot && ring_batch < B)) return DFLASH_ERR_SHAPE;
  if (!feats || !n_new || !ctx_len || !ring_k || !ring_v) return DFLASH_ERR_ARG;
  if (!aligned(feats, 16) || !aligned(ring_k, 16) || !aligned(ring_v, 16) || !aligned(n_new, 4) ||
      !aligned(ctx_len, 8) || (req_slot && !aligned(req_slot, 4)))
    return DFLASH_ERR_ALIGN;
  if (!aligned(workspace, 256)) return DFLASH_ERR_WORKSPACE;
  AppendWs ws = append_layout(h, workspace);
  if (ws_bytes < ws.bytes) return DFLASH_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GemmScratch scratch{ws.gemm_partial, kGemmPartialFloats, ws.gemm_counters, kGemmCounters, ws.status,
                      h->num_sms};
  const int M = B * n_max;
  const int d = c.hidden;
  const int Kc = c.n_feat * c.feat_dim;
  int rc;

  // With token tiles of at most 32 the RMSNorm that forms H_t is folded into
  // the two GEMMs: W_c's epilogue writes fp16(H * g_c) and per-tile sums of
  // squares of H, the K/V GEMM scales by rstd (GemmRowScale) and rotates keys
  // at their positions itself.  Otherwise W_c writes fp32 H and a separate
  // RMSNorm (which also tabulates the rotations) normalises it.
  const bool fold = gemm_token_tile(M) <= 32;
  const int d_tiles = (d + 127) / 128;
  {
    GemmAMaps A;
    A.map[0] = h->w_c;
    GemmEpi e = epi_base(fold ? EPI_NORM_IN : EPI_F32, M, d, fold ? nullptr : ws.fused, d, ws.status);
    if (fold) {
      e.xg = static_cast<__half*>(ws.ht);
      e.xg_g = static_cast<const float*>(h->w.g_c);
      e.ssq = ws.ssq;
    }
    const int nt = d_tiles;
    rc = launch_gemm(A, single_map(), nt, feats, OPND_BF16, M, Kc, e, scratch, splits_for(h, nt, M, Kc),
                     s, true);
    if (rc) return rc;
  }
  if (!fold) {
    rc = launch_rmsnorm_rope(ws.fused, M, d, static_cast<const float*>(h->w.g_c), c.eps, 0, ws.ht,
                             ws.status, ctx_len, n_max, ws.rope_cs, c.head_dim / 2, h->rope, s);
    if (rc) return rc;
  }
  GemmRowScale rsc;
  rsc.ssq = ws.ssq;
  rsc.parts = d_tiles;
  rsc.n = d;
  rsc.eps = c.eps;
  // K/V of every layer into the ring, up to kMaxAMaps layers per launch
  const int kvd = c.n_kv_heads * c.head_dim;
  const int tiles_per_layer = 2 * kvd / 128;
  for (int l0 = 0; l0 < c.n_layers; l0 += kMaxAMaps) {
    const int nl = c.n_layers - l0 < kMaxAMaps ? c.n_layers - l0 : kMaxAMaps;
    GemmAMaps A;
    for (int i = 0; i < nl; ++i) A.map[i] = h->maps[l0 + i].qkv;
    GemmAOpts ao = single_map();
    for (int i = 0; i < nl; ++i) ao.scale[i] = h->layers[l0 + i].s_qkv;
    ao.n_maps = nl;
    ao.tiles_per_map = tiles_per_layer;
    ao.row_offset = c.n_q_heads * c.head_dim;
    GemmEpi e = epi_base(EPI_KV_RING, M, nl * 2 * kvd, nullptr, 0, ws.status);
    e.ctx_len = ctx_len;
    e.rope_cs = fold ? nullptr : ws.rope_cs;
    e.rope_inv = h->rope;
    e.hd = c.head_dim;
    e.ring_k = ring_k;
    e.ring_v = ring_v;
    e.ring_batch = ring_batch;
    e.window = c.window;
    e.n_kv = c.n_kv_heads;
    e.kv_dim = kvd;
    e.n_max = n_max;
    e.n_new = n_new;
    e.req_slot = req_slot;
    e.layer0 = l0;
    const int nt = nl * tiles_per_layer;
    rc = launch_gemm(A, ao, nt, ws.ht, h->wtype, M, d, e, scratch, splits_for(h, nt, M, d), s, true,
                     fold ? &rsc : nullptr);
    if (rc) return rc;
  }
  return launch_add_lengths(B, n_new, ctx_len, s);
}

int dflash_draft_block(dflash_handle* h, int B, int gamma, const int32_t* anchor,
                       const int64_t* ctx_len, const int32_t* req_slot, const void* ring_k,
                       const void* ring_v, int ring_batch, int topk, const dflash_sampling* sampling,
                       const dflash_draft_out* out, void* workspace, size_t ws_bytes,
                       dflash_stream_t stream) {
  if (!h || !out) return DFLASH_ERR_ARG;
  const dflash_config& c = h->cfg;
  if (B < 1 || B > c.batch_max || gamma < 2 || gamma > c.gamma_max) return DFLASH_ERR_SHAPE;
  if (topk < 0 || topk > c.topk_max || topk > c.vocab) return DFLASH_ERR_SHAPE;
  if (ring_batch < 1 || (!req_slot && ring_batch < B)) return DFLASH_ERR_SHAPE;
  if (!anchor || !ctx_len || !ring_k || !ring_v) return DFLASH_ERR_ARG;
  if (topk == 0 && (out->topk_ids || out->topk_vals)) return DFLASH_ERR_ARG;
  if (sampling) {
    if (!(sampling->temperature > 0.0f) || !(sampling->top_p > 0.0f) || !(sampling->top_p <= 1.0f) ||
        !sampling->seeds || !out->q)
      return DFLASH_ERR_ARG;
    if (!aligned(sampling->seeds, 8) || !aligned(out->q, 4)) return DFLASH_ERR_ALIGN;
  } else if (out->q) {
    return DFLASH_ERR_ARG;
  }
  if (!aligned(ring_k, 16) || !aligned(ring_v, 16) || !aligned(anchor, 4) || !aligned(ctx_len, 8) ||
      (req_slot && !aligned(req_slot, 4)))
    return DFLASH_ERR_ALIGN;
  const void* outs[] = {out->topk_ids, out->topk_vals, out->lse, out->logits, out->draft};
  for (const void* p : outs)
    if (p && !aligned(p, 4)) return DFLASH_ERR_ALIGN;
  if (!aligned(workspace, 256)) return DFLASH_ERR_WORKSPACE;
  DraftWs ws = draft_layout(h, workspace);
  if (ws_bytes < ws.bytes) return DFLASH_ERR_WORKSPACE;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GemmScratch scratch{ws.gemm_partial, kGemmPartialFloats, ws.gemm_counters, kGemmCounters, ws.status,
                      h->num_sms};
  h->prof_used = 0;
  const int M = B * gamma;
  const int R = B * (gamma - 1);
  const int d = c.hidden, hd = c.head_dim;
  const int qd = c.n_q_heads * hd;
  const int qkv_dim = (c.n_q_heads + 2 * c.n_kv_heads) * hd;
  const size_t ring_layer = (size_t)ring_batch * c.n_kv_heads * c.window * hd;
  int rc;

  int slot = prof_begin(h, s);
  rc = launch_embed_norm(h->w.embed, anchor, B, gamma, h->mask_id, c.vocab, d,
                         static_cast<const float*>(h->layers[0].g_attn), c.eps, ws.x, ws.h, ws.status,
                         ctx_len, ws.rope_cs, hd / 2, h->rope, s);
  if (rc) return rc;
  prof_end(h, s, slot, (double)M * d * (2 + 4 + 4), DFLASH_KIND_NORM);
  AttnArgs aa;
  aa.qkv = static_cast<const __half*>(ws.qkv);
  aa.ld_qkv = qkv_dim;
  aa.out = static_cast<__half*>(ws.attn);
  aa.ld_out = qd;
  aa.ctx_len = ctx_len;
  aa.req_slot = req_slot;
  aa.gamma = gamma;
  aa.n_q = c.n_q_heads;
  aa.n_kv = c.n_kv_heads;
  aa.hd = hd;
  aa.window = c.window;
  aa.ring_batch = ring_batch;
  aa.splits = attn_splits(h, B);
  aa.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)hd));
  aa.status = ws.status;
  // ring K/V of the visible window + block q, k, v read, output written
  double attn_bytes = 0.0;
  {
    const double win = c.window;  // upper bound; the visible part is min(L, W) per request
    attn_bytes = (double)B * c.n_kv_heads * win * hd * 2 * 2 + (double)M * (qkv_dim + qd) * 2;
  }

  // With many tokens a GEMM tile's residual read-modify-write stalls its
  // epilogue: O and down then store their fp32 output and the RMSNorm that
  // follows (which reads the row anyway) adds it to the stream.  With few
  // tokens the epilogue adds it itself and the latency-bound RMSNorm reads
  // one array.
  const bool defer = M > kFreeResidTokens;
  // With token tiles of at most 32 there is no RMSNorm launch: the O and down
  // epilogues write the next GEMM's input fp16(x * g) and per-tile sums of
  // squares of the updated stream, and the next GEMM scales its outputs by the
  // norm's rstd (GemmRowScale).
  const bool fuse_norm = !defer && gemm_token_tile(M) <= 32;
  const int d_tiles = (d + 127) / 128;
  GemmRowScale rsc;
  rsc.ssq = ws.ssq;
  rsc.parts = d_tiles;
  rsc.n = d;
  rsc.eps = c.eps;
  const double ssq_bytes = fuse_norm ? 4.0 * d_tiles * M : 0.0;
  // bytes per weight element streamed (E4M3 codes: 1, plus a 4-byte scale per row)
  const double wb = h->wtype == OPND_E4M3 ? 1.0 : 2.0;
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerMaps& lm = h->maps[l];
    const dflash_layer_weights& L = h->layers[l];
    {  // QKV (+RoPE on q and k)
      GemmAMaps A;
      A.map[0] = lm.qkv;
      const GemmAOpts ao = single_map(L.s_qkv);
      GemmEpi e = epi_base(EPI_QKV, M, qkv_dim, ws.qkv, qkv_dim, ws.status);
      e.ctx_len = ctx_len;
      e.gamma = gamma;
      e.rope_cs = ws.rope_cs;
      e.rope_rows = (c.n_q_heads + c.n_kv_heads) * hd;
      e.hd = hd;
      const int nt = (qkv_dim + 127) / 128;
      // layer 0 reads the embedding's RMSNorm; later layers fold theirs in
      const bool rs_here = fuse_norm && l > 0;
      rc = draft_gemm(h, A, ao, nt, ws.h, M, d, e, scratch, s,
                      wb * qkv_dim * d + 2.0 * M * d + 2.0 * M * qkv_dim + (rs_here ? ssq_bytes : 0.0),
                      rs_here ? &rsc : nullptr);
      if (rc) return rc;
    }
    slot = prof_begin(h, s);
    rc = launch_attention(static_cast<const char*>(ring_k) + l * ring_layer * 2,
                          static_cast<const char*>(ring_v) + l * ring_layer * 2, aa, B, s);
    if (rc) return rc;
    prof_end(h, s, slot, attn_bytes, DFLASH_KIND_ATTENTION);
    {  // O projection (+ residual, here or in the next RMSNorm)
      GemmAMaps A;
      A.map[0] = lm.o;
      GemmEpi e = defer ? epi_base(EPI_F32, M, d, ws.y, d, ws.status)
                        : epi_base(EPI_RESID, M, d, ws.x, d, ws.status);
      if (fuse_norm) {  // the MLP's RMSNorm input and sums of squares
        e.ssq = ws.ssq;
        e.xg = static_cast<__half*>(ws.h);
        e.xg_g = static_cast<const float*>(L.g_mlp);
      }
      const int nt = (d + 127) / 128;
      rc = draft_gemm(h, A, single_map(L.s_o), nt, ws.attn, M, qd, e, scratch, s,
                      wb * d * qd + 2.0 * M * qd + (defer ? 4.0 : 8.0) * M * d +
                          (fuse_norm ? 2.0 * M * d + ssq_bytes : 0.0));
      if (rc) return rc;
    }
    if (!fuse_norm) {
      slot = prof_begin(h, s);
      rc = launch_add_rmsnorm(ws.x, defer ? ws.y : nullptr, 1, M, d, static_cast<const float*>(L.g_mlp),
                              c.eps, 0, ws.h, ws.status, s);
      if (rc) return rc;
      prof_end(h, s, slot, (double)M * d * (defer ? 14 : 6), DFLASH_KIND_NORM);
    }
    {  // gate | up + SwiGLU
      GemmAMaps A;
      A.map[0] = lm.gate;
      A.map[1] = lm.up;
      GemmAOpts ao = single_map(L.s_gate);
      ao.n_maps = 2;
      ao.dual = 1;
      ao.scale[1] = L.s_up;
      GemmEpi e = epi_base(EPI_SWIGLU, M, c.ffn, ws.mlp, c.ffn, ws.status);
      const int nt = c.ffn / 64;
      rc = draft_gemm(h, A, ao, nt, ws.h, M, d, e, scratch, s,
                      2.0 * wb * c.ffn * d + 2.0 * M * d + 2.0 * M * c.ffn + ssq_bytes,
                      fuse_norm ? &rsc : nullptr);
      if (rc) return rc;
    }
    {  // down (+ residual, here or in the next RMSNorm)
      GemmAMaps A;
      A.map[0] = lm.down;
      GemmEpi e = defer ? epi_base(EPI_F32, M, d, ws.y, d, ws.status)
                        : epi_base(EPI_RESID, M, d, ws.x, d, ws.status);
      if (fuse_norm) {  // the next layer's (or the final) RMSNorm input and sums of squares
        e.ssq = ws.ssq;
        e.xg = static_cast<__half*>(ws.h);
        e.xg_g = static_cast<const float*>(l + 1 < c.n_layers ? h->layers[l + 1].g_attn : h->w.g_final);
      }
      const int nt = (d + 127) / 128;
      rc = draft_gemm(h, A, single_map(L.s_down), nt, ws.mlp, M, c.ffn, e, scratch, s,
                      wb * d * c.ffn + 2.0 * M * c.ffn + (defer ? 4.0 : 8.0) * M * d +
                          (fuse_norm ? 2.0 * M * d + ssq_bytes : 0.0));
      if (rc) return rc;
    }
    if (fuse_norm) continue;
    slot = prof_begin(h, s);
    const float* add = defer ? ws.y : nullptr;
    if (l + 1 < c.n_layers)
      rc = launch_add_rmsnorm(ws.x, add, 1, M, d, static_cast<const float*>(h->layers[l + 1].g_attn),
                              c.eps, 0, ws.h, ws.status, s);
    else  // the final RMSNorm reads only the MASK rows; the stream is not needed after it
      rc = launch_add_rmsnorm(ws.x, add, 0, R, d, static_cast<const float*>(h->w.g_final), c.eps,
                              gamma, ws.hf, ws.status, s);
    if (rc) return rc;
    prof_end(h, s, slot, (double)(l + 1 < c.n_layers ? M : R) * d * (defer ? 14 : 6), DFLASH_KIND_NORM);
  }
  // Top-k, log-sum-exp and the top-1 draft.  When the caller wants fp32
  // logits or sampling needs them, the LM head writes them and a chunked
  // top-k kernel reads them back.  Otherwise the logits are never written:
  // the LM head's epilogue keeps each vocabulary tile's top keys and (max,
  // sum of exp) per MASK row and a merge kernel finishes.  Measured on
  // GB300 with logits written in both: the epilogue's top-k costs the LM head
  // more than the separate kernel takes (batch 1: +22 us against 15 us;
  // batch 32, gamma 8: +83 us against 98 us).
  float* logits = out->logits ? out->logits : (sampling ? ws.logits : nullptr);
  const bool fused_topk = logits == nullptr;
  const int k_eff = topk > 0 ? topk : 1;
  const int vtiles = (c.vocab + 127) / 128;
  const int slots = topk_slots(c.topk_max);
  const double part_bytes = (double)R * vtiles * (8.0 * k_eff + 8.0);
  {  // shared LM head on the gamma - 1 MASK rows
    GemmAMaps A;
    A.map[0] = h->lm_head;
    const double logit_bytes = logits ? 4.0 * R * c.vocab : part_bytes;
    GemmEpi e = epi_base(EPI_F32, fuse_norm ? M : R, c.vocab, logits, c.vocab, ws.status);
    if (fused_topk) {
      e.tk_keys = ws.tk_keys;
      e.tk_ml = ws.tk_ml;
      e.tk_slots = slots;
      e.tk_k = k_eff;
      e.tk_tiles = vtiles;
    }
    if (fuse_norm) {
      // the final RMSNorm folded in: all M rows of the stream in (the anchors
      // share the token tile), the MASK rows out
      e.out_gather = gamma;
      rc = draft_gemm(h, A, single_map(h->w.s_lm_head), vtiles, ws.h, M, d, e, scratch, s,
                      wb * c.vocab * d + 2.0 * M * d + logit_bytes + ssq_bytes, &rsc);
    } else {
      rc = draft_gemm(h, A, single_map(h->w.s_lm_head), vtiles, ws.hf, R, d, e, scratch, s,
                      wb * c.vocab * d + 2.0 * R * d + logit_bytes);
    }
    if (rc) return rc;
  }
  slot = prof_begin(h, s);
  int32_t* ids_out = topk > 0 ? out->topk_ids : nullptr;
  float* vals_out = topk > 0 ? out->topk_vals : nullptr;
  int32_t* draft_out = sampling ? nullptr : out->draft;
  if (fused_topk)
    rc = launch_topk_merge(R, vtiles, slots, k_eff, ws.tk_keys, ws.tk_ml, ids_out, vals_out, out->lse,
                           draft_out, s);
  else
    rc = launch_topk_lse(logits, R, c.vocab, k_eff, ws.topk_keys, ws.topk_ml, ws.topk_counters, ids_out,
                         vals_out, out->lse, draft_out, s);
  if (rc) return rc;
  prof_end(h, s, slot, fused_topk ? part_bytes : 4.0 * R * c.vocab, DFLASH_KIND_TOPK);
  if (sampling) {
    slot = prof_begin(h, s);
    rc = launch_probs(R, c.vocab, logits, sampling->temperature, sampling->top_p, out->q, s);
    if (rc) return rc;
    prof_end(h, s, slot, 8.0 * R * c.vocab, DFLASH_KIND_SAMPLING);
    if (out->draft) {
      rc = launch_sample_rows(R, c.vocab, out->q, c.vocab, gamma - 1, sampling->seeds, sampling->step,
                              0u, out->draft, gamma - 1, ws.samp_counters, ws.samp_zsum, ws.status, s);
      if (rc) return rc;
    }
  }
  return DFLASH_OK;
}

}  // extern "C"
