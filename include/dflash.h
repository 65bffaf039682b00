/*
 * dflash.h — C ABI of libdflash.so: single-pass block drafting with target
 * context injection, plus lossless verification, on one GB300 (sm_103a).
 *
 * What the library computes (sources are the three pages it follows):
 *   - "DFlash vs DFlash 2" (blog), section "Conditioning on the target model":
 *       H_t = RMSNorm(W_c [H^(l1); ...; H^(l5)]),
 *       Q_i = W^Q_i H_d,  K_i = [W^K_i H_t ; W^K_i H_d],  V_i = [W^V_i H_t ; W^V_i H_d];
 *     target features enter only through keys and values; block positions
 *     attend to one another non-causally.
 *   - same page, section "DFlash: generate the block all at once": one
 *     masked, bidirectional pass over [anchor, MASK, MASK, ...] through a
 *     small stack of Qwen-style layers, shared embedding and LM head.
 *   - same page, section "The problem: one expensive token at a time":
 *     greedy verification accepts drafts that match the target's choice;
 *     sampled verification accepts y ~ q with probability min(1, p(y)/q(y)),
 *     resamples from the normalised [p - q]+ at the first rejection and emits
 *     a bonus token from the target's next distribution when every draft
 *     survives.
 *   - "Speculative decoding" (product doc), section "How it works", and the
 *     model card "Beam-1.0-501B-A23B-DFlash2", section "Model": a 4,096-token
 *     sliding window over the context, top candidates kept per position,
 *     5 layers, hidden 5120, 40 query / 8 KV heads of dim 128, SwiGLU 17,408,
 *     vocabulary 151,936.
 *
 * Conventions this library fixes where the pages are silent:
 *   - RoPE (rotate-half pairs (j, j + hd/2), inv_freq_j = theta^(-2j/hd)) on
 *     queries and keys at absolute positions; context keys are stored rotated.
 *   - Pre-norm layers; RMSNorm(x) = x / sqrt(mean(x^2) + eps) * g; SwiGLU MLP
 *     W_down(silu(W_gate h) * W_up h); final RMSNorm before the LM head.
 *   - A context of length L (positions 0..L-1 have target features) puts the
 *     block at positions L..L+gamma-1; the context key at position s is visible
 *     iff L - W <= s < L; block row j >= 1 predicts the token at L + j, so the
 *     LM head runs on the gamma - 1 MASK rows.
 *   - Randomness: Philox-4x32-10 keyed by a per-request 64-bit seed, counter
 *     (step_lo, step_hi, position, purpose), purpose 0 = draft draw, 1 = accept
 *     test, 2 = residual / bonus draw.  Accept iff (u24 * 2^-24) * q(y) < p(y)
 *     evaluated exactly; every draw is an integer inverse CDF over
 *     floor(weight * 2^45).
 *
 * Arithmetic.  The drafter's matrices arrive as bf16.  dflash_create copies
 * the five matrices of every layer and the LM head into one fp16 buffer of the
 * handle: every bf16 value of magnitude 2^-14 .. 65504 is exactly an fp16
 * value, and smaller ones keep an absolute error below 2^-25.  Every
 * contraction of the draft pass then runs on fp16 operands with fp32
 * accumulation, and the activations between kernels are stored as fp16:
 * 11 significant bits where bf16 keeps 8, at the same tensor-core rate.  An
 * activation beyond the fp16 range sets DFLASH_ERR_RANGE in the workspace
 * status word.  W_c and the target features stay bf16 (the features are
 * bf16 as given), and so does the context K/V ring.
 *
 * Memory and ownership.  Every pointer argument, unless it says "host", is
 * device memory owned by the caller.  With bf16 weights dflash_create
 * allocates the handle's fp16 matrix copy (2 bytes per element of those
 * matrices; dflash_destroy frees it); with E4M3 weights the handle holds no
 * device memory.  No other call allocates device memory, except the
 * benchmark hook dflash_profile_enable.  Calls other than
 * create/destroy are asynchronous on the given stream, never synchronise the
 * host, and may be captured into a CUDA graph.
 *
 * Workspace.  draft_block, ctx_append, probs and verify take a caller-owned
 * device workspace of at least the size the matching *_workspace_bytes
 * function returns, 256-byte aligned, ZERO-FILLED BEFORE ITS FIRST USE.  The
 * library leaves the workspace's counter region zeroed after every call, so
 * it can be reused without clearing.  The first 4 bytes of every workspace are
 * a device status word: 0, or a DFLASH_ERR_* code written by a kernel (for
 * example a bounded wait that gave up).  Calls that share one workspace must
 * not overlap on the GPU.
 *
 * Errors.  Every function returns DFLASH_OK (0) or a negative DFLASH_ERR_*
 * code after validating its arguments on the host; nothing is launched when
 * validation fails.  No C++ exception crosses this boundary.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dflash_stream_t; /* a cudaStream_t */

enum {
  DFLASH_OK = 0,
  DFLASH_ERR_ARG = -1,            /* null pointer or invalid scalar argument */
  DFLASH_ERR_SHAPE = -2,          /* sizes out of range or inconsistent */
  DFLASH_ERR_ALIGN = -3,          /* a pointer is not 16-byte aligned */
  DFLASH_ERR_UNSUPPORTED = -4,    /* a configuration the kernels do not cover */
  DFLASH_ERR_LAUNCH = -5,         /* a kernel launch failed */
  DFLASH_ERR_DEVICE_TIMEOUT = -6, /* device status: a bounded wait gave up */
  DFLASH_ERR_WORKSPACE = -7,      /* workspace missing or too small */
  DFLASH_ERR_CUDA = -8,           /* a CUDA runtime / driver call failed */
  DFLASH_ERR_RANGE = -9           /* a weight or (device status) an activation is beyond
                                     the fp16 range */
};

enum { DFLASH_VERIFY_GREEDY = 0, DFLASH_VERIFY_SAMPLED = 1 };

/* Drafter dimensions.  Constraints checked by dflash_create: head_dim is 64
 * or 128; hidden, ffn, n_q_heads*head_dim and n_feat*feat_dim are multiples
 * of 64; hidden <= 12288; n_q_heads is a multiple of n_kv_heads; 2 <= gamma_max <= 16;
 * (n_q_heads / n_kv_heads) * gamma_max <= 128 (the query rows of one KV head);
 * 1 <= topk_max <= 16; window >= 1. */
typedef struct dflash_config {
  int hidden;      /* d */
  int n_q_heads;   /* Hq */
  int n_kv_heads;  /* Hkv */
  int head_dim;    /* hd */
  int ffn;         /* SwiGLU width F */
  int vocab;       /* V */
  int n_layers;    /* NL */
  int n_feat;      /* number of target layers read (5) */
  int feat_dim;    /* width of each target feature */
  int window;      /* W, sliding-window length of the context cache */
  int gamma_max;   /* largest block size any call will use */
  int topk_max;    /* largest per-position top-k any call will use */
  int batch_max;   /* largest B any draft_block / ctx_append call will use */
  int append_max;  /* largest rows per request of one ctx_append call */
  float rope_theta;
  float eps;
  int mask_id;     /* MASK token id; -1 selects vocab - 1 */
  int weight_format; /* DFLASH_WEIGHTS_BF16 (0) or DFLASH_WEIGHTS_E4M3 (1) */
} dflash_config;

/* Storage of the drafter's matrices (w_qkv, w_o, w_gate, w_up, w_down of
 * every layer, and lm_head).  BF16: bf16 values, copied by dflash_create into
 * an fp16 buffer of the handle.  E4M3: FP8 codes (1 sign, 4 exponent bits
 * with bias 7, 3 mantissa bits, no infinities, largest finite 448) with one
 * float32 scale per output row, weight[r][c] = code[r][c] * scale[r]; used in
 * place (the handle holds no copy), half the bytes a draft pass streams.  The
 * pages serve their models in bf16, FP8 and NVFP4 ("Speculative decoding"
 * product doc, introduction; model card, section "Serve") without fixing the
 * FP8 format; dflash_quantize_e4m3 makes such weights from bf16 ones. */
enum { DFLASH_WEIGHTS_BF16 = 0, DFLASH_WEIGHTS_E4M3 = 1 };

/* One drafter layer.  Matrices are bf16 row-major [out, in] (the torch Linear
 * layout), gains are float32.  All device pointers, 16-byte aligned. */
typedef struct dflash_layer_weights {
  const void* g_attn; /* float32 [d] */
  const void* w_qkv;  /* bf16 [(Hq + 2 Hkv) hd, d]: q rows, then k rows, then v rows */
  const void* w_o;    /* bf16 [d, Hq hd] */
  const void* g_mlp;  /* float32 [d] */
  const void* w_gate; /* bf16 [F, d] */
  const void* w_up;   /* bf16 [F, d] */
  const void* w_down; /* bf16 [d, F] */
  /* E4M3 weights only: float32 scale of every output row of the matrix above
   * of the same name ([(Hq + 2 Hkv) hd], [d], [F], [F], [d]); else NULL */
  const float* s_qkv;
  const float* s_o;
  const float* s_gate;
  const float* s_up;
  const float* s_down;
} dflash_layer_weights;

typedef struct dflash_weights {
  const void* embed;   /* bf16 [V, d], shared with the target */
  const void* lm_head; /* bf16 [V, d], shared with the target */
  const void* w_c;     /* bf16 [d, n_feat * feat_dim] */
  const void* g_c;     /* float32 [d], gain of the RMSNorm that forms H_t */
  const void* g_final; /* float32 [d] */
  const dflash_layer_weights* layers; /* HOST array of n_layers entries */
  const float* s_lm_head; /* E4M3 weights only: float32 [V] row scales of lm_head */
} dflash_weights;

typedef struct dflash_handle dflash_handle;

/* Validate cfg, record the weight pointers and encode the TMA descriptors.
 * BF16 weights: copy w_qkv, w_o, w_gate, w_up, w_down of every layer and
 * lm_head into the handle's fp16 buffer (allocated here), which the draft
 * pass then reads; the copied matrices need not stay alive.  E4M3 weights:
 * nothing is copied; the codes and scales are read in place and must stay
 * alive and unchanged while the handle is used, like embed, w_c and the
 * gains in both formats.  Synchronises the device (the weights may have
 * been written on any stream).  Must be called with the weights' device
 * current.  Returns DFLASH_OK and *out, or an error (then *out is NULL):
 * DFLASH_ERR_RANGE if a copied bf16 matrix holds a value beyond +-65504 (or a
 * NaN), or an E4M3 matrix a NaN code or a scale that is not finite and
 * positive; DFLASH_ERR_ARG if an E4M3 scale pointer is missing;
 * DFLASH_ERR_CUDA if a buffer cannot be allocated. */
int dflash_create(const dflash_config* cfg, const dflash_weights* w, dflash_handle** out);
int dflash_destroy(dflash_handle* h);

/* Bytes of workspace each call needs for the handle's limits. */
size_t dflash_draft_workspace_bytes(const dflash_handle* h);
size_t dflash_append_workspace_bytes(const dflash_handle* h);
size_t dflash_verify_workspace_bytes(int batch, int gamma, int vocab);
size_t dflash_probs_workspace_bytes(int rows, int vocab);

/* Context injection ("Conditioning on the target model": H_t equation and the
 * K/V injection equation).  For every request b and row j < n_new[b]:
 *   pos = ctx_len[b] + j,
 *   H_t = RMSNorm(W_c concat(feats[b, j, 0..nf-1, :])),
 *   for each layer i: ring_k[i, slot(b), :, pos mod W, :] = RoPE(W^K_i H_t, pos),
 *                     ring_v[i, slot(b), :, pos mod W, :] = W^V_i H_t,
 * then ctx_len[b] += n_new[b].  Rows j >= n_new[b] are ignored.  To append
 * only the last W positions of a long prompt, set ctx_len[b] to the position
 * of the first appended row before the call.
 *   B            requests in this call, 1..batch_max
 *   n_max        rows per request in feats, 1..append_max
 *   feats        bf16 [B, n_max, n_feat, feat_dim]
 *   n_new        int32 [B], each in [0, n_max]
 *   ctx_len      int64 [B], in/out
 *   req_slot     int32 [B] ring row of each request, or NULL for slot(b) = b
 *   ring_k/v     bf16 [n_layers, ring_batch, Hkv, W, hd]
 */
int dflash_ctx_append(dflash_handle* h, int B, int n_max, const void* feats,
                      const int32_t* n_new, int64_t* ctx_len, const int32_t* req_slot,
                      void* ring_k, void* ring_v, int ring_batch,
                      void* workspace, size_t ws_bytes, dflash_stream_t stream);

/* Sampling parameters of draft_block (host struct).  temperature > 0. */
typedef struct dflash_sampling {
  float temperature;     /* logits are divided by it before the softmax */
  float top_p;           /* nucleus mass in (0, 1]; 1 disables it */
  const uint64_t* seeds; /* device [B] Philox keys, one per request */
  uint64_t step;         /* Philox step (counter words 0-1) */
} dflash_sampling;

/* Outputs of draft_block (host struct of device pointers; NULL = not wanted). */
typedef struct dflash_draft_out {
  int32_t* topk_ids; /* int32 [B, gamma-1, topk], descending logit, ties to lower id */
  float* topk_vals;  /* float32 [B, gamma-1, topk] logits of those ids */
  float* lse;        /* float32 [B, gamma-1] log-sum-exp of each row's logits */
  float* logits;     /* float32 [B, gamma-1, V] raw logits */
  float* q;          /* float32 [B, gamma-1, V] q = top_p(softmax(logits / T));
                        requires sampling */
  int32_t* draft;    /* int32 [B, gamma-1] proposed tokens: the top-1 id, or
                        with sampling y ~ q (Philox purpose 0, position j) */
} dflash_draft_out;

/* One single-pass block draft per request ("DFlash: generate the block all at
 * once"; "Conditioning on the target model").  Block ids are
 * [anchor[b], MASK x (gamma-1)] at positions ctx_len[b] .. ctx_len[b]+gamma-1;
 * every layer attends over [visible context window ; whole block].
 *   B          1..batch_max;  gamma 2..gamma_max;  topk 0..topk_max
 *   anchor     int32 [B];  ctx_len int64 [B] (0 allowed: the block alone)
 *   req_slot   int32 [B] or NULL;  ring_k/v as in ctx_append
 *   sampling   host pointer or NULL (greedy drafting)
 * Device status (dflash_read_status): DFLASH_ERR_RANGE if an fp16 activation
 * between kernels would exceed +-65504.  With B * gamma <= 32 the layers'
 * RMSNorms are folded into the GEMMs around them and one of those activations
 * is the unnormalised residual stream times the norm's gains.
 */
int dflash_draft_block(dflash_handle* h, int B, int gamma, const int32_t* anchor,
                       const int64_t* ctx_len, const int32_t* req_slot,
                       const void* ring_k, const void* ring_v, int ring_batch, int topk,
                       const dflash_sampling* sampling, const dflash_draft_out* out,
                       void* workspace, size_t ws_bytes, dflash_stream_t stream);

/* Sampling distribution of raw logits: probs = top_p(softmax(logits / T)),
 * renormalised (model card "Beam-1.0-501B-A23B-DFlash2", section "Acceptance
 * length": temperature 0.7, top-p 0.99).  Nucleus: ids ordered by
 * (probability desc, id asc), the shortest prefix whose mass reaches top_p.
 *   logits, probs  float32 [rows, V] (may not alias) */
int dflash_probs(int rows, int vocab, const float* logits, float temperature, float top_p,
                 float* probs, void* workspace, size_t ws_bytes, dflash_stream_t stream);

/* The drafter's proposal y ~ q ("The problem: one expensive token at a time":
 * the drafter proposes y from its distribution q): for request b and
 * position i < G, y[b, i] is the fixed-point inverse-CDF draw from q[b, i]
 * with Philox (seeds[b], step, position i, purpose 0).  draft_block makes the
 * same draw when given sampling parameters.
 *   q  float32 [B, G, V], rows normalised;  y  int32 [B, G] out */
int dflash_sample_draft(int B, int G, int vocab, const float* q, const uint64_t* seeds,
                        uint64_t step, int32_t* y, void* workspace, size_t ws_bytes,
                        dflash_stream_t stream);
size_t dflash_sample_workspace_bytes(int rows, int vocab);

/* Verification ("The problem: one expensive token at a time").
 *   mode GREEDY:  target = target logits float32 [B, gamma, V]; q, seeds unused.
 *                 n = longest prefix with draft[b, i] == argmax target[b, i]
 *                 (ties to the lowest id); tokens[n] = argmax target[b, n].
 *   mode SAMPLED: target = p float32 [B, gamma, V], q float32 [B, gamma-1, V],
 *                 rows normalised; accept draft i iff
 *                 (u24_i * 2^-24) q_i(y_i) < p_i(y_i) (Philox purpose 1,
 *                 position i); at the first rejection j draw from
 *                 max(0, p_j - q_j) (float32), or from p_j if that has zero
 *                 mass; if all survive draw the bonus from p_{gamma-1}
 *                 (Philox purpose 2, position n).
 *   draft      int32 [B, gamma-1]
 *   accept_len int32 [B] out: n in [0, gamma-1]; tau = n + 1
 *   tokens     int32 [B, gamma] out: drafts 0..n-1, the correction or bonus
 *              at n, -1 after.
 *   next_anchor, n_append  int32 [B] out, each may be NULL: the commit step
 *              of the cycle ("Speculative decoding" product doc, section "How
 *              it works": accepted tokens are emitted, then the next block) —
 *              next_anchor = tokens[b, n] (the anchor of the next block) and
 *              n_append = n + 1 (the positions the target has now scored: the
 *              anchor and the n accepted drafts, whose features ctx_append
 *              takes next). */
int dflash_verify(int mode, int B, int gamma, int vocab, const float* target, const float* q,
                  const int32_t* draft, const uint64_t* seeds, uint64_t step,
                  int32_t* accept_len, int32_t* tokens, int32_t* next_anchor, int32_t* n_append,
                  void* workspace, size_t ws_bytes, dflash_stream_t stream);

/* Benchmark hook.  dflash_profile_enable(h, n) allocates a device buffer of
 * n + 1 timestamps (n = 0 frees it); afterwards every draft_block call on h
 * launches, on the call's stream, a one-warp mark kernel before its first
 * launch and after each of its first n launches.  A mark lets the next kernel
 * start early (programmatic dependent launch) as it would without it, waits
 * for the launch before it to complete and writes the device clock
 * (%globaltimer).  dflash_profile_read synchronises the device and returns,
 * for each launch of the last call, the time from the previous launch's
 * completion to its own in ms (these add up to the whole pass, overlap
 * between neighbouring kernels included), its algorithmic bytes (operands
 * read + results written, each counted once) and its kind (DFLASH_KIND_*);
 * *count receives the number of launches (<= cap).  A draft_block call
 * captured into a CUDA graph captures its marks too, so a replayed graph can
 * be profiled (read after the replay). */
enum { DFLASH_KIND_GEMM = 0, DFLASH_KIND_ATTENTION = 1, DFLASH_KIND_NORM = 2,
       DFLASH_KIND_TOPK = 3, DFLASH_KIND_SAMPLING = 4 };
int dflash_profile_enable(dflash_handle* h, int n_pairs);
int dflash_profile_read(dflash_handle* h, float* ms, double* bytes, int* kinds, int cap, int* count);

/* Verification for callers that cannot provide device memory.  The pages have
 * no counterpart to this entry point: it exists for callers that cannot
 * allocate or lend device memory at the point where they verify — for example
 * a serving process whose device memory is reserved up front by another
 * allocator, where a further cudaMalloc would fail or fragment the
 * reservation, or a host framework that forbids plug-ins from allocating
 * device memory (cudaMalloc also synchronises the device).
 *
 * Same arguments and results as dflash_verify, without the workspace: the
 * kernels' scratch (status word, per-request tickets, argmax keys, chunk
 * masses) lives in one fixed 256 KiB __device__ array inside this library,
 * which every GPU that loads the library holds until the process exits.  The
 * call allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine); it clears the part of the array that must start at zero with an
 * asynchronous memset on the given stream.
 *   Limit: 256 + 256*ceil(4B/256) + 256*ceil(8*B*gamma/256)
 *          + 16*B*ceil(vocab/8192) bytes (rounded up to 256) must not exceed
 *          256 KiB: at gamma 16 and vocabulary 151,936 the largest B is 600
 *          (B = 601 needs 262,656 bytes); larger calls return
 *          DFLASH_ERR_SHAPE, launch nothing and leave the outputs untouched.
 *   A call made outside any stream capture looks up the array's device
 *   address with the current device (cudaGetSymbolAddress) and remembers it
 *   with the current context.  A call made while its stream is captured uses
 *   that remembered address, so the first call on a device, and the first
 *   after a device reset, must be made before any capture; a captured call
 *   without one returns DFLASH_ERR_UNSUPPORTED and launches nothing.
 *   Every call on a device shares the one array and the array keeps the last
 *   call's contents: calls whose work overlaps on the GPU (two streams, or
 *   graphs replayed concurrently) race on it and must be serialised by the
 *   caller.  Device-side errors go to the array's status word, which callers
 *   of this entry point cannot read back; use dflash_verify for that. */
int dflash_verify_noalloc(int mode, int B, int gamma, int vocab, const float* target,
                          const float* q, const int32_t* draft, const uint64_t* seeds,
                          uint64_t step, int32_t* accept_len, int32_t* tokens,
                          int32_t* next_anchor, int32_t* n_append, dflash_stream_t stream);

/* E4M3 weights from bf16 ones (the format of DFLASH_WEIGHTS_E4M3), one CTA
 * per row: scale[r] = max_c |w[r][c]| / 448 in float32 (1 for a row of
 * zeros); code[r][c] = w[r][c] / scale[r] (float32 division, round to
 * nearest) rounded to the nearest E4M3 value, ties to an even mantissa,
 * saturating at +-448.  A NaN or infinite weight makes NaN codes, which
 * dflash_create refuses.  The pages fix no FP8 scheme; this is the
 * library's reading (see DFLASH_WEIGHTS_E4M3).
 *   w       bf16 [rows, cols], cols a multiple of 16, 16-byte aligned
 *   codes   uint8 [rows, cols] out, 16-byte aligned
 *   scales  float32 [rows] out
 * Asynchronous on the stream; allocates nothing. */
int dflash_quantize_e4m3(const void* w, int rows, int cols, void* codes, float* scales,
                         dflash_stream_t stream);

/* Copy the workspace status word to the host (synchronises the stream). */
int dflash_read_status(const void* workspace, int32_t* status_host, dflash_stream_t stream);

const char* dflash_strerror(int code);

/* Self-test of the bounded-wait machinery every pipelined kernel uses: one
 * CTA waits on a shared-memory mbarrier that nothing arrives on, gives up
 * after `limit_ns` nanoseconds (clamped to 1 s) and writes
 * DFLASH_ERR_DEVICE_TIMEOUT into the workspace status word.  The GPU context
 * stays usable.  workspace: >= 256 bytes, its status word is overwritten. */
int dflash_selftest_timeout(void* workspace, long long limit_ns, dflash_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H_ */
