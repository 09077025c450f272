/*
 * qd.h — C ABI of libqd.so: the token-decode step of a Qwen3-style GQA
 * transformer on one GB300 (sm_103a).
 *
 * Sources (page title, section):
 *   [KL-DEC]  "GPU Kernel Lab" README, "Decode integration": the order of one
 *             decode step (fixed token/position buffers, projections, Q/K
 *             RMSNorm + RoPE + direct K/V cache write, GQA split-KV attention,
 *             residual + RMSNorm, gate/up GEMV + SwiGLU, residual + next
 *             RMSNorm, LM-head GEMV + argmax + token/position update, CUDA
 *             graph replay).
 *   [KL-FUN]  "GPU Kernel Lab" README, "Fundamental kernels": Qwen-exact RMSNorm
 *             cast order, RoPE pair rotation, SwiGLU, stable softmax,
 *             warp-reduced decode GEMV, split-KV decode attention.
 *   [CD-GEMV] "qwen3-8b-rtx4080-cutedsl" README, "Decode GEMV path".
 *   [CD-ATT]  "qwen3-8b-rtx4080-cutedsl" README, "GQA + QK-Norm" and
 *             "Split-KV decode attention".
 *   [CD-ROPE] "qwen3-8b-rtx4080-cutedsl" README, "RoPE vectorized kernel" and
 *             "L2 persistence" (the RoPE frequency table).
 *   [CD-GRAPH] "qwen3-8b-rtx4080-cutedsl" README, "CUDA graphs".
 *   [EQ-SPEED] "emit_qwen38_generate" rustdoc, "Where the speed comes from":
 *             one GEMV per shared activation (concatenated rows), one graph per
 *             token with the token and position advanced on device, residual +
 *             RMSNorm + activation re-quantisation fused, Q8_0 lanes (deq).
 *   [KL-PAGED] "GPU Kernel Lab" README, "Measured final results" / "Serving
 *             system": K/V in fixed physical pages read through a page table.
 *
 * Conventions shared by every call:
 *   - Return value: QD_OK (0) or a negative QD_ERR_* code; qd_last_error()
 *     returns a thread-local message for the last failure of this thread.
 *   - All tensor pointers are DEVICE pointers owned by the caller, unless a
 *     parameter says "host". Pointers must be 16-byte aligned.
 *   - Every call is asynchronous on the given cudaStream_t (0 = legacy default
 *     stream); none synchronises the host, allocates memory or reads device
 *     memory on the host, except qd_check_device_error and the qd_graph_* calls
 *     documented as such. Arguments are validated on the host before any launch;
 *     on an error nothing is launched.
 *   - Matrices are row-major. bf16 = IEEE bfloat16, f16 = IEEE binary16, f32 =
 *     binary32. "Rows" are output features, "cols" the reduction dimension.
 *   - Device-side range faults (a page id outside the cache, a position past
 *     the cache capacity, an all-NaN logit row, a full out_tokens buffer) do not
 *     trap: the kernel skips the access and sets a sticky error word that
 *     qd_check_device_error reports.
 */
#ifndef QD_H
#define QD_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  QD_OK = 0,
  QD_ERR_INVALID_ARG = -1,
  QD_ERR_UNSUPPORTED = -2,
  QD_ERR_CUDA = -3,
  QD_ERR_WORKSPACE = -4,
  QD_ERR_DEVICE = -5, /* a sticky device-side range fault was recorded */
};

/* device error word bits (qd_check_device_error) */
enum {
  QD_DEVERR_PAGE = 1,      /* page id >= n_pages or logical page >= max_pages */
  QD_DEVERR_POS = 2,       /* position >= cache capacity */
  QD_DEVERR_NAN = 4,       /* an all-NaN logit row in argmax */
  QD_DEVERR_STEPS = 8,     /* step >= max_steps in argmax_advance */
  QD_DEVERR_TIMEOUT = 16,  /* a bounded wait on an asynchronous copy gave up */
};

/* Weight formats: BF16; Q8_0 (32-wide int8 blocks with an fp16 scale); INT4 (W4A16: */
/* 4-bit codes with one fp16 scale per output row, see qd_gemv_w4).                  */
typedef enum { QD_W_BF16 = 0, QD_W_Q8_0 = 1, QD_W_INT4 = 2 } qd_wtype;
/* Q8_0 activation lanes ([EQ-SPEED] ``deq``): F32 = dequantising lane,
 * I8 = activation re-quantised per 32-block to int8 (dp4a lane). */
typedef enum { QD_ACT_F32 = 0, QD_ACT_I8 = 1 } qd_act;

const char* qd_last_error(void);
int qd_version(void);

/* ------------------------------------------------------------------------ */
/* Weight-streaming GEMV, BF16 weights ([CD-GEMV], [KL-FUN] "warp-reduced     */
/* decode GEMV", [EQ-SPEED] item 1).                                          */
/*   y[b, r] = sum_c W[r, c] * x[b, c]      b < batch, r < rows, c < cols      */
/* W: bf16 [rows, cols]. x: bf16 [batch, cols] (x_is_f32 = 0) or f32            */
/* [batch, cols] (x_is_f32 = 1; the kernel rounds x to bf16 first). y: f32      */
/* [batch, rows]. Accumulation in f32, deterministic order.                   */
/* batch 1: CUDA-core ring GEMV (cols % 8 == 0). batch 2..8 with bf16 x and     */
/* cols % 32 == 0: the weight-streaming GEMV with its multiply-add on mma.sync   */
/* (each weight read once for all rows); otherwise batch <= 8 runs the CUDA-core */
/* GEMV (QD_SMALLB_IMPL=simt forces it). batch >= 9: the product is a dense     */
/* contraction and runs on the tcgen05 tensor cores ("qwen3-8b-rtx4080-         */
/* cutedsl" README, "Baseline tiled GEMM"), one CTA per 128 rows x 64 batch     */
/* rows; above 128 batch rows (a prompt's tokens, for prefill) a persistent     */
/* kernel, one CTA per SM over 128 x 256 tiles (QD_GEMM_WIDE=tiles: one CTA per */
/* tile). Needs bf16 x and cols % 64 == 0.                                      */
int qd_gemv_bf16(const void* W, int rows, int cols, const void* x, int x_is_f32,
                 float* y, int batch, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Q8_0 GEMV, both lanes ([EQ-SPEED] ``deq``).                                 */
/* W = f32(d[r, c/32]) * qs[r, c]; qs: int8 [rows, cols]; d: f16 [rows, cols/32]. */
/* act == QD_ACT_F32: y[r] = sum_b f32(d[r,b]) * sum_i qs[r,32b+i] * x_f32[32b+i] */
/* act == QD_ACT_I8:  y[r] = sum_b f32(d[r,b]) * f32(x_d[b]) * (int32 block dot  */
/*                    of qs and x_q), the int32 dot exact.                      */
/* Unused activation pointers may be NULL. Limits: cols % 32 == 0.             */
int qd_gemv_q8_0(const int8_t* qs, const void* d_f16, int rows, int cols,
                 const float* x_f32, const int8_t* x_q, const void* x_d_f16,
                 qd_act act, float* y, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Batched Q8_0 projection on the tcgen05 tensor cores ("qwen3-8b-rtx4080-     */
/* cutedsl" README, "Baseline tiled GEMM"; Q8_0 blocks per [EQ-SPEED]):          */
/*   y[b, r] = sum_c bf16(f32(d[r, c/32]) * qs[r, c]) * x[b, c]                  */
/* Each weight is widened on chip to bf16 (the product is exact in binary32,     */
/* then one round to nearest even) and the contraction runs as bf16 MMA with f32 */
/* accumulation. qs: int8 [rows, cols]; d: f16 [rows, cols/32]; x: bf16          */
/* [batch, cols]; y: f32 [batch, rows]. workspace: NULL (no K split) or device   */
/* scratch of qd_gemm_workspace_bytes(rows, cols, QD_W_Q8_0) bytes, zero-filled  */
/* before its first use (each call leaves it zero-filled); with it, grids that   */
/* do not fill the SMs split K and sum the partials in split order.              */
/* Limits: cols % 256 == 0, batch >= 1 (above 64: 64-row tiles, no K split and   */
/* the workspace unused), every pointer 16-byte aligned.                         */
size_t qd_gemm_workspace_bytes(int rows, int cols, qd_wtype wtype);
int qd_gemm_q8_0(const int8_t* qs, const void* d_f16, int rows, int cols, const void* x_bf16,
                 int batch, float* y, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* W4A16 GEMV ("GPU Kernel Lab" README, "Quantization experiments": W4A16 decode */
/* GEMV, packed INT4 LM head with local top-k, per-output-channel weight          */
/* quantization; "qwen3-8b-rtx4080-cutedsl" README, "W4A16 dequant-fused GEMM").   */
/* W: uint8 [rows, cols/2], each byte two offset-binary nibbles u = q + 8 (q in    */
/* [-8, 7]), the even column in the low nibble; d: f16 [rows], one scale per row:  */
/* w[r, c] = f32(d[r]) * q[r, c].  y[r] = sum_c w[r, c] * x[c] with x bf16 [cols];  */
/* y f32 [rows]; batch 1, f32 accumulation. Limits: cols % 32 == 0, cols <= 16384; */
/* W and x 16-byte aligned, d 2-byte aligned.                                      */
int qd_gemv_w4(const uint8_t* W, const void* d_f16, int rows, int cols, const void* x_bf16, float* y,
               cudaStream_t stream);
/* The same with a workspace: with cols % 256 == 0 the product runs on the tcgen05  */
/* tensor cores (each weight code widened to bf16 in tensor memory, the activation */
/* as the other operand), and a matrix whose 128-row tiles underfill the SMs      */
/* splits K across CTAs, adding the partials in split order. workspace: NULL (no  */
/* split; what qd_gemv_w4 does) or zero-filled device scratch of                  */
/* qd_gemv_w4_workspace_bytes(rows, cols) bytes (0: no split), left zero-filled.  */
size_t qd_gemv_w4_workspace_bytes(int rows, int cols);
int qd_gemv_w4_ex(const uint8_t* W, const void* d_f16, int rows, int cols, const void* x_bf16, float* y,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream);
/* The INT4 LM-head form: y as qd_gemv_w4 (the logits), and the top k rows of y     */
/* (value descending, the lower row first among equal values, NaN never chosen):  */
/* topk_ids int32 [k] (-1 past the non-NaN rows), topk_vals f32 [k]. Each CTA picks */
/* the top k of its rows; the last CTA merges them. 1 <= k <= 16. workspace:        */
/* zero-filled device scratch of qd_w4_topk_workspace_bytes() bytes, left zero.   */
size_t qd_w4_topk_workspace_bytes(void);
int qd_gemv_w4_topk(const uint8_t* W, const void* d_f16, int rows, int cols, const void* x_bf16, int k,
                    float* y, int32_t* topk_ids, float* topk_vals, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream);

/* Activation re-quantisation per 32-block ([EQ-SPEED] item 3): amax = max|x|,  */
/* d = amax / 127, q = round-half-away(x * (1/d)) in IEEE binary32 (0 if d = 0), */
/* d stored as f16 (round to nearest even). x: f32 [n]; x_q: int8 [n];            */
/* x_d: f16 [n/32]. Limits: n % 32 == 0.                                        */
int qd_quantize_q8_0(const float* x, int n, int8_t* x_q, void* x_d_f16, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* GQA split-KV decode attention over a paged cache ([CD-ATT], [KL-FUN],       */
/* [KL-PAGED]).                                                               */
/*   out[b, h, :] = sum_{t < seq_lens[b]} softmax_t(scale * q[b,h,:].K_b[t,g,:]) */
/*                  * V_b[t, g, :],   g = h / (n_q_heads / n_kv_heads)          */
/* q: f32 [batch, n_q_heads, head_dim]. k_pages, v_pages: bf16                  */
/* [n_pages, n_kv_heads, page_size, head_dim]; logical token t of sequence b    */
/* lives in page page_table[b * max_pages + t / page_size], slot t % page_size. */
/* page_table: int32 [batch, max_pages]. seq_lens: int32 [batch] (device).      */
/* out: f32 [batch, n_q_heads, head_dim]. workspace: device scratch of at least  */
/* qd_attn_workspace_bytes(...) bytes, zero-filled before its first use (the   */
/* call leaves it zero-filled again). seq_lens[b] == 0 gives out = 0.           */
/* Limits: head_dim == 128, n_q_heads % n_kv_heads == 0, n_q_heads/n_kv_heads   */
/* <= 8, page_size >= 1, seq_lens[b] <= max_pages * page_size.                  */
size_t qd_attn_workspace_bytes(int batch, int n_q_heads, int n_kv_heads, int max_ctx);
int qd_attn_decode_paged(const float* q, const void* k_pages, const void* v_pages,
                         const int32_t* page_table, const int32_t* seq_lens, int batch,
                         int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                         int max_pages, int n_pages, float scale, float* out,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Allocation-free variant of qd_attn_decode_paged. (The pages describe no    */
/* such call; it exists for callers that cannot allocate device memory:       */
/* hosts whose device memory is reserved up front by their own pool, plugins  */
/* handed only input and output buffers, and latency-critical loops where     */
/* cudaMalloc/cudaFree would add an implicit device synchronisation.)          */
/* Same arguments, layouts and result as qd_attn_decode_paged, without the    */
/* workspace: the split-KV scratch is a static 8 MiB device array inside the  */
/* library, held by every GPU that loads it until the process exits. Shapes   */
/* whose workspace (qd_attn_workspace_bytes) exceeds 8 MiB are rejected with  */
/* QD_ERR_WORKSPACE. The call allocates nothing; it clears the scratch's      */
/* ticket counters with cudaMemsetAsync on `stream` before the launch. The    */
/* first call on each device looks up the array's device address            */
/* (cudaGetSymbolAddress) with that device current; make that first call     */
/* before any stream capture. All calls share the one array, which keeps the  */
/* last call's contents: calls that overlap on the GPU (for example on two     */
/* streams) race on it and must be serialised by the caller.                 */
int qd_attn_decode_paged_noalloc(const float* q, const void* k_pages, const void* v_pages,
                                 const int32_t* page_table, const int32_t* seq_lens, int batch,
                                 int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                                 int max_pages, int n_pages, float scale, float* out,
                                 cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Greedy argmax + on-device advance ([KL-DEC] "LM-head GEMV + argmax +        */
/* token/position update"; [EQ-SPEED] item 2).                                  */
/* For each b < batch: t = lowest index of the maximum of logits[b, :vocab]     */
/* (NaN never wins; an all-NaN row gives 0 and sets QD_DEVERR_NAN);             */
/* out_tokens[b * max_steps + step[b]] = t (if step[b] < max_steps, else        */
/* QD_DEVERR_STEPS); tok[b] = t; pos[b] += 1; step[b] += 1.                      */
/* workspace: zero-filled scratch of qd_argmax_workspace_bytes(batch) bytes.    */
size_t qd_argmax_workspace_bytes(int batch);
int qd_argmax_advance(const float* logits, int vocab, int batch, int32_t* tok, int32_t* pos,
                      int32_t* step, int32_t* out_tokens, int max_steps, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* RoPE cos/sin table ([CD-ROPE]): table[p, i] = (cos(p * f_i), sin(p * f_i)),  */
/* f_i = theta^(-2i/head_dim), i < head_dim/2, p < max_pos; angles evaluated in  */
/* binary64 on the device, stored as f32 pairs. table: f32 [max_pos, head_dim/2, 2]. */
int qd_rope_table_init(float* table, int max_pos, int head_dim, float theta, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Layers and the whole decode step.                                         */
typedef struct {
  int hidden, n_q_heads, n_kv_heads, head_dim, ffn;
  float rms_eps, rope_theta;
  qd_wtype wtype;
  qd_act act; /* Q8_0 models only */
} qd_layer_dims;

/* Row order ([EQ-SPEED] item 1): w_qkv = [q rows (Hq*D); k rows (Hkv*D);       */
/* v rows (Hkv*D)] x hidden; w_o = hidden x (Hq*D); w_gu = [gate rows (ffn);     */
/* up rows (ffn)] x hidden; w_down = hidden x ffn. BF16: bf16 matrices, s_* NULL. */
/* Q8_0: int8 matrices plus f16 scales [rows, cols/32]. INT4: packed matrices    */
/* [rows, cols/2] (as qd_gemv_w4) plus f16 scales [rows]. Norm weights: bf16.     */
typedef struct {
  const void *w_qkv, *w_o, *w_gu, *w_down;
  const void *s_qkv, *s_o, *s_gu, *s_down;
  const void *ln_in, *ln_post, *q_norm, *k_norm;
} qd_layer_weights;

typedef struct qd_layer qd_layer; /* opaque: dims + pointers, no tensor data */

/* Validates and records dims and pointers (host memory only; the weights stay */
/* owned by the caller and must outlive the handle).                          */
int qd_create_layer(const qd_layer_dims* dims, const qd_layer_weights* w, qd_layer** out);
int qd_destroy_layer(qd_layer* layer);

/* One decode token for `batch` sequences ([KL-DEC]):                          */
/*   res = embed[tok]; per layer: xn = RMSNorm(res; ln_in) (Qwen cast order);  */
/*   [q;k;v] = W_qkv xn; q,k = RoPE_pos(RMSNorm_head(q; q_norm / k; k_norm));    */
/*   K/V cache slot pos = (k, v) in bf16; o = GQA attention over slots 0..pos;  */
/*   res += W_o bf16(o); xn = RMSNorm(res; ln_post); [g;u] = W_gu xn;           */
/*   res += W_down bf16(silu(g) * u); then logits = W_lm RMSNorm(res; final_norm) */
/*   and argmax_advance (tok, pos, step, out_tokens updated on the device).     */
/* k_cache / v_cache: arrays (host memory) of n_layers device pointers, each    */
/* bf16 [n_pages, n_kv_heads, page_size, head_dim]. A contiguous cache is one   */
/* page of max_ctx tokens per sequence (page_size = max_ctx, page_table[b] = b). */
/* tok, pos, step: int32 [batch] device; out_tokens: int32 [batch, max_steps].   */
/* rope_table: from qd_rope_table_init with max_pos >= every position reached.  */
/* logits: f32 [batch, vocab] device output. workspace: device scratch of        */
/* qd_step_workspace_bytes(args) bytes, zero-filled before first use.           */
/* BF16 layers: batch 1 runs the ring GEMV path. Batch 2..8 with a bf16 LM head  */
/* and hidden, n_q_heads * head_dim, ffn multiples of 32 runs every projection   */
/* on the mma.sync weight-streaming GEMV (five launches per layer, RMSNorm and   */
/* SwiGLU fused). Batch 9..64 (and 3..8 with QD_SMALLB_IMPL=tc, from           */
/* QD_TC_MIN_BATCH, default 3) runs every projection as a tcgen05 GEMM over the  */
/* batch when those dims are multiples of 64; otherwise batch <= 8 runs the      */
/* CUDA-core GEMV path (batch 2: K <= 12288).                                    */
/* Q8_0 layers: batch 1 runs the                                                 */
/* Q8_0 GEMV lanes (act, lm_act); 2..64 runs the tcgen05 GEMMs with the weights  */
/* widened to bf16 as in qd_gemm_q8_0 (act and lm_act unused; dims % 256 == 0,   */
/* scales 16-byte aligned). INT4 layers: batch 1, the W4A16 GEMVs with bf16      */
/* activations (dims % 32 == 0, <= 16384).                                       */
/* LM head: lm_wtype QD_W_INT4 with lm_head_scales = the per-row f16 scales is an */
/* INT4 head (batch 1): its GEMV also picks the top_k tokens (0: only the argmax)  */
/* into topk_ids / topk_vals [top_k] and advances the step itself. Otherwise the  */
/* head is Q8_0 when lm_head_scales is set, else bf16, followed by argmax_advance. */
typedef struct {
  const qd_layer* const* layers;
  int n_layers;
  const void* embed;           /* bf16 [vocab, hidden] */
  const void* final_norm;      /* bf16 [hidden] */
  const void* lm_head;         /* bf16 [vocab, hidden], or int8 for a Q8_0 head */
  const void* lm_head_scales;  /* f16 [vocab, hidden/32] for a Q8_0 head, else NULL */
  qd_act lm_act;               /* Q8_0 head lane */
  int vocab;
  void* const* k_cache;
  void* const* v_cache;
  const int32_t* page_table;
  int page_size, max_pages, n_pages;
  const float* rope_table;
  int rope_max_pos;
  int32_t *tok, *pos, *step, *out_tokens;
  int max_steps;
  int batch;
  float* logits;
  void* workspace;
  size_t workspace_bytes;
  qd_wtype lm_wtype;   /* QD_W_INT4 for an INT4 head (see above) */
  int top_k;           /* INT4 head: 0..16 tokens into topk_ids / topk_vals */
  int32_t* topk_ids;
  float* topk_vals;
} qd_step_args;

size_t qd_step_workspace_bytes(const qd_step_args* args);
int qd_decode_step(const qd_step_args* args, cudaStream_t stream);

/* Whole-step CUDA graph ([CD-GRAPH], [EQ-SPEED] item 2): captures
 * `steps_per_launch` consecutive qd_decode_step calls (the token and position
 * advance on the device, so replays need no host round trip) on `stream`, and
 * instantiates the graph. Capture happens on the calling thread; the args
 * (pointers and sizes) are frozen into the graph. qd_graph_launch replays it on
 * `stream`. qd_graph_create synchronises nothing but must not be called while
 * `stream` is already capturing. */
typedef struct qd_graph qd_graph;
int qd_graph_create(const qd_step_args* args, int steps_per_launch, cudaStream_t stream,
                    qd_graph** out);
int qd_graph_launch(qd_graph* g, cudaStream_t stream);
int qd_graph_destroy(qd_graph* g);

/* ------------------------------------------------------------------------ */
/* Speculative verify ("qwen3-8b-rtx4080-cutedsl" README, "Speculative          */
/* decoding": a draft proposes tokens and the target model checks k of them in  */
/* one forward pass that reuses the weight bytes already streamed). For the one */
/* sequence of `args` (batch 1): the k input tokens are tok[0] (the last token   */
/* emitted) and draft[0 .. k-2], at positions pos[0] .. pos[0] + k - 1. They run  */
/* as k rows of one pass: every projection streams its weights once for the k   */
/* rows (bf16: the mma.sync GEMV when the dims are multiples of 32; Q8_0, or     */
/* QD_SMALLB_IMPL=tc: tcgen05 GEMMs); the                                        */
/* k new K/V rows are written to the cache first, and row i attends to positions */
/* 0 .. pos[0] + i (causal among the drafted tokens).                           */
/* Outputs: logits f32 [k, vocab] (device, 16-byte aligned); target int32 [k]:   */
/* the argmax of each row (the model's token after input i, as in               */
/* qd_argmax_advance); n_accept int32 [1]: m = the number of leading drafts with  */
/* draft[i] == target[i] (0 <= m <= k - 1). The state advances on the device:     */
/* out_tokens[step .. step + m] = draft[0 .. m - 1], target[m]; tok = target[m];  */
/* pos += m + 1; step += m + 1. Cache rows past pos[0] + m hold the rejected      */
/* drafts' K/V until a later step overwrites them.                               */
/* draft: int32 [k - 1] device (may be NULL when k == 1). 1 <= k <= 8. The       */
/* projections' K must be multiples of 32 (bf16 on the mma.sync GEMV), 64 (bf16 */
/* on tcgen05) or 256 (Q8_0, whose weights are                                   */
/* widened on chip as in qd_gemm_q8_0). workspace: args->workspace of at least    */
/* qd_verify_workspace_bytes(args, k) bytes, zero-filled before first use; the   */
/* pass's scratch follows the first qd_step_workspace_bytes(args) bytes (the      */
/* decode step's, left untouched), so passes and decode steps may alternate.     */
size_t qd_verify_workspace_bytes(const qd_step_args* args, int k);
int qd_verify_step(const qd_step_args* args, const int32_t* draft, int k, float* logits, int32_t* target,
                   int32_t* n_accept, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Prefill ("qwen3-8b-rtx4080-cutedsl" README, "Flash Attention 2" and           */
/* "Baseline tiled GEMM": the prompt is processed as one batch of rows with      */
/* tiled attention that never forms the full score matrix). For the one sequence */
/* of `args` (batch 1): tokens int32 [n_tokens] (device) sit at positions         */
/* pos[0] .. pos[0] + n_tokens - 1. Every layer runs over all rows at once: the   */
/* projections are tcgen05 GEMMs over 64- or 256-token tiles (Q8_0 weights above */
/* 128 rows widened to bf16 once per projection, bf16(f32(d) q), into the        */
/* workspace first), the rows' K/V are                                           */
/* written to the cache first, and row i attends causally to positions 0 ..       */
/* pos[0] + i (the keys already cached included) on tcgen05 (QD_PREFILL_ATTN=mma: */
/* the mma.sync kernel). The workspace includes a packed copy of the kv heads'    */
/* keys up to the cache capacity (and, for Q8_0 above 128 rows, the bf16 copy of */
/* the largest projection). The last row alone goes through the final            */
/* norm and the LM head: logits f32 [vocab] (device, 16-byte aligned). The state  */
/* then advances as one decode step from the last row: tok = argmax (first index */
/* among equal maxima), out_tokens[step] = tok, pos += n_tokens, step += 1.      */
/* Position errors (pos[0] + n_tokens past the cache or the RoPE table) set      */
/* QD_DEVERR_POS. 1 <= n_tokens <= 32768; BF16 or Q8_0 weights (K multiples of 64 */
/* or 256 as in qd_verify_step). workspace: args->workspace of at least           */
/* qd_prefill_workspace_bytes(args, n_tokens) bytes, zero-filled before first use; */
/* as in qd_verify_step, the decode step's part of it is left untouched.          */
size_t qd_prefill_workspace_bytes(const qd_step_args* args, int n_tokens);
int qd_prefill(const qd_step_args* args, const int32_t* tokens, int n_tokens, float* logits, cudaStream_t stream);

/* Reads and clears the sticky device error word (synchronises `stream`).      */
/* *bits receives a mask of QD_DEVERR_*. Returns QD_OK or QD_ERR_CUDA.           */
int qd_check_device_error(cudaStream_t stream, int* bits);

/* Number of kernel launches one qd_decode_step call issues for these args.    */
int qd_step_launch_count(const qd_step_args* args);

/* ------------------------------------------------------------------------ */
/* Test-only exports (make the bit-exactness claims directly checkable).      */
/* qd_debug_q8_block_dots runs the production Q8_0 GEMV of the i8 lane          */
/* (qd_gemv_q8_0 with act = QD_ACT_I8 and x_q, x_d given: the same dispatch and  */
/* kernels as the decode step's Q8_0 GEMVs) in a form that also stores each      */
/* int32 block dot it forms: dots[r, b] = sum_i qs[r, 32b+i] * x_q[32b+i],        */
/* int32 [rows, cols/32]; y: f32 [rows], the GEMV result.                        */
int qd_debug_q8_block_dots(const int8_t* qs, const void* d_f16, int rows, int cols, const int8_t* x_q,
                           const void* x_d_f16, int32_t* dots, float* y, cudaStream_t stream);
/* idx[b, t] = page_table[b*max_pages + t/page_size]*page_size + t%page_size for */
/* t < n_tokens: the physical token slot the attention kernels read, through    */
/* the same device function they use. A page id outside [0, n_pages) gives      */
/* idx = -1 and sets QD_DEVERR_PAGE (the attention kernels read page 0 there).  */
int qd_debug_paged_indices(const int32_t* page_table, int batch, int max_pages,
                           int page_size, int n_pages, int n_tokens, int32_t* idx,
                           cudaStream_t stream);
/* The timeout path of the kernels' bounded waits: one thread arms an mbarrier   */
/* for bytes no copy will deliver (none is issued) and waits on it for limit_us  */
/* microseconds (1 .. 1000000); the wait gives up, sets QD_DEVERR_TIMEOUT and the */
/* kernel returns, leaving the context usable. Asynchronous on `stream`.          */
int qd_debug_wait_timeout(int limit_us, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QD_H */
