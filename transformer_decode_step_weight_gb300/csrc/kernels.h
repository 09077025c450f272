// Internal launcher interface between the C-ABI layer (api.cu) and the kernel
// translation units. Host-only declarations; no CUDA device code here.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qd {

struct DevInfo {
  int sm_count;
  int max_smem_optin;
};
const DevInfo& dev_info();

// Launch options shared by every kernel launch of a decode step.
struct Launch {
  cudaStream_t stream;
  bool pdl;          // programmatic dependent launch attribute
  int trig_late;     // 1: let the next kernel launch only near the end of this one
  int* err;          // sticky device error word
};

// ----------------------------------------------------------------- L2 prefetch plan
// Weights of a later GEMV, cut the way every GEMV cuts its rows over the grid
// (span c = rows [c * rows_base + min(c, rows_extra), ...) is one CTA's), of
// which the leading `head_bytes` of every span are fetched into L2 by a kernel
// that runs before that GEMV and leaves DRAM idle part of its time. A hint
// only: nothing waits on it and nothing depends on it for correctness.
struct L2Prefetch {
  const void* base;               // null: nothing to fetch
  unsigned long long row_bytes;   // a multiple of 16
  int rows_base, rows_extra, n_spans;
  unsigned long long head_bytes;  // per span; >= the span's bytes fetches all of it
};
// The plan for an R-row matrix read by a GEMV (same partition as the GEMV
// launchers); head_bytes = ~0 fetches the whole matrix. Null plan when the row
// pitch or the base is not 16-byte aligned.
L2Prefetch l2_plan_rows(const void* base, int R, size_t row_bytes, size_t head_bytes);

// ----------------------------------------------------------------- GEMV bf16
enum GemvPro { PRO_X_BF16 = 0, PRO_X_F32 = 1, PRO_RMSNORM = 2, PRO_SWIGLU = 3 };
// EPI_SWIGLU (batch-1 ring form only): W holds [gate (F rows); up (F rows)] and the
// output is h = bf16(silu(gate . x) * (up . x)) [F] in y_bf16. Each CTA takes the
// same pair range of both halves, so gate_j and up_j meet in one CTA.
// EPI_TOPK (INT4 LM head): y = logits; the launch's top-k tokens and, when tok is set,
// the argmax advance of the step (see GemvW4Args).
enum GemvEpi { EPI_STORE = 0, EPI_RESID_ADD = 1, EPI_SWIGLU = 2, EPI_TOPK = 3 };

struct GemvBf16Args {
  const void* W;          // bf16 [R, K]
  int R, K, batch;
  int pro;                // GemvPro
  const void* x;          // PRO_X_BF16: bf16 [batch, K]; PRO_X_F32: f32 [batch, K];
                          // PRO_RMSNORM: f32 residual [batch, K]; PRO_SWIGLU: f32 [batch, 2K]
  const void* norm_w;     // bf16 [K] (PRO_RMSNORM)
  float eps;
  int epi;                // GemvEpi
  float* y;               // f32 [batch, R]
  L2Prefetch pf;          // batch-1 ring form: weights of the next GEMV, fetched once
                          // this CTA's own copies are all issued (zero: none)
  int ring_kb;            // batch-1 ring form: ring size in KB (0: the default)
  void* y_bf16;           // EPI_SWIGLU: bf16 [R / 2]
  int w_evict_first;      // batch-1 ring form: weight copies marked evict-first in L2
};
bool gemv_bf16_supported(int K, int batch);
// True when a batch-1 GEMV of K columns takes the ring form, and when that form
// can also take EPI_SWIGLU.
bool gemv_bf16_ring_ok(int K, int batch);
bool gemv_bf16_swiglu_ok(int K);
cudaError_t launch_gemv_bf16(const GemvBf16Args& a, const Launch& L);

// ----------------------------------------------------------------- GEMV W4A16 (INT4 weights)
// W: packed rows [R, K / 2] (two offset-binary nibbles q + 8 per byte, even column
// low), d: fp16 [R] per-row scales; y[r] = f32(d[r]) * sum_c q[r, c] x[c] with bf16
// activations x. Prologues and epilogues as the BF16 GEMV (batch 1). EPI_SWIGLU:
// y_bf16 [R / 2] = bf16(silu(gate) * up). EPI_TOPK: y [R] = logits, topk_ids / vals
// [top_k] (value descending, lower row first, NaN never chosen; -1 past the non-NaN
// rows) and, when tok is set, tok = the first of them, out_tokens[step] = tok,
// pos += 1, step += 1 (all-NaN logits: token 0 and QD_DEVERR_NAN). ws: zero-filled
// scratch of w4_topk_workspace_bytes() bytes, left zero-filled.
struct GemvW4Args {
  const void* W;
  const void* d;
  int R, K;
  int pro;
  const void* x;
  const void* norm_w;
  float eps;
  int epi;
  float* y;
  void* y_bf16;
  int w_evict_first;
  L2Prefetch pf;
  int top_k;
  void* ws;
  int32_t *tok, *pos, *step, *out_tokens;
  int max_steps;
  int32_t* topk_ids;
  float* topk_vals;
  void* split_ws;         // tcgen05 form: split-K partials and tickets (null: no split)
  size_t split_ws_bytes;
};
bool gemv_w4_supported(int K);
size_t w4_topk_workspace_bytes();
cudaError_t launch_gemv_w4(const GemvW4Args& a, const Launch& L);
// The tcgen05 form (gemv_w4_tc.cu): K % 256 == 0, K <= 16384. `ws` (zero-filled
// before first use, left so) lets tiles that underfill the SMs split K; null: no split.
bool gemv_w4_tc_supported(int K);
size_t gemv_w4_tc_workspace_bytes(int R, int K, bool pair);
cudaError_t launch_gemv_w4_tc(const GemvW4Args& a, void* ws, size_t ws_bytes, const Launch& L);
// Tensor map of a row-major uint8 [rows, cols_bytes] matrix: boxes of 128 bytes x
// box_rows rows, 128-byte swizzle (CUtensorMap storage, 128 bytes, 128-byte aligned).
cudaError_t encode_tmap_u8_sw128(void* map, const void* base, uint64_t rows, uint64_t cols_bytes, uint32_t box_rows);

// ----------------------------------------------------------------- batched GEMM (tcgen05)
struct GemmTcArgs {
  const void* W;          // bf16 [R, K], or Q8_0 int8 values [R, K] when S is set
  const void* S;          // Q8_0 fp16 scales [R, K/32], or null (bf16 W)
  const void* X;          // bf16 [B, K]
  int R, K, B;            // B <= 64, or more rows in 64-token tiles (no K split)
  int epi;                // GemvEpi
  float* y;               // f32 [B, R]
  void* ws;               // split-K partials and tile tickets (zero-filled before first use,
  size_t ws_bytes;        // left so); null: no split
};

// Weight-streaming GEMV over B <= 8 activation rows on mma.sync (gemv_mma.cu).
struct GemvMmaArgs {
  const void* W;          // bf16 [R, K]; EPI_SWIGLU: [gate F rows; up F rows], R = 2F
  int R, K, B;            // K % 32 == 0, 1 <= B <= 8
  int pro;                // PRO_X_BF16: x bf16 [B, K]; PRO_RMSNORM: x f32 [B, K], norm_w bf16 [K]
  const void* x;
  const void* norm_w;
  float eps;
  int epi;                // EPI_STORE / EPI_RESID_ADD: y f32 [B, R]; EPI_SWIGLU: y_bf16 [B, F]
  float* y;
  void* y_bf16;
  int w_evict_first;
  L2Prefetch pf;          // weights of the next GEMV, fetched once this CTA's copies are issued
};
bool gemv_mma_supported(int R, int K, int B);
cudaError_t launch_gemv_mma(const GemvMmaArgs& a, const Launch& L);

bool gemm_tc_supported(int R, int K, int B);
bool gemm_tc_q8_supported(int R, int K, int B);
// B > 64 rows (prefill): token tiles over grid z, no K split; B <= 64: the forms above.
bool gemm_tc_rows_supported(int R, int K, int B, bool q8);
// Tensor map (CUtensorMap, 128-byte aligned storage of 128 bytes) of a row-major
// bf16 [rows, cols] matrix: boxes of box_rows x 64 columns, 128-byte swizzle.
cudaError_t encode_tmap_bf16_2d(void* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
// K splits a launch of this shape takes, and the workspace they need.
int gemm_tc_splits(int R, int K, bool q8 = false);
size_t gemm_tc_workspace_bytes(int R, int K, bool q8 = false);
cudaError_t launch_gemm_tc(const GemmTcArgs& a, const Launch& L);
// Prefill gate+up (BF16, more than 128 rows): h[t, j] = bf16(silu(g) u) with g = row j
// and u = row F + j of W [2F, K] applied to X [B, K] bf16, written to h [B, F] bf16.
bool gemm_tc_swiglu_supported(int F, int K, int B);
cudaError_t launch_gemm_tc_swiglu(const void* W, const void* X, int F, int K, int B, void* h, const Launch& L);
// Q8_0 matrix (int8 [R, K], fp16 scales [R, K / 32]) widened to bf16 [R, K], each weight
// bf16(f32(d) * q); K a multiple of 32, W and out 16-byte aligned.
cudaError_t launch_q8_widen(const void* W, const void* S, int R, int K, void* out, const Launch& L);

// row-wise helpers of the batched step
cudaError_t launch_rmsnorm_rows(const float* x, const void* w, int B, int K, float eps, void* out_bf16,
                                const Launch& L);
cudaError_t launch_swiglu_rows(const float* gu, int B, int F, void* out_bf16, const Launch& L);

// ----------------------------------------------------------------- GEMV Q8_0
struct GemvQ8Args {
  const int8_t* qs;       // int8 [R, K]
  const void* d;          // f16 [R, K/32]
  int R, K;
  int act;                // 0 = f32 lane, 1 = i8 lane
  int pro;                // GemvPro (PRO_X_BF16 not used)
  const void* x;          // f32 x / residual / gu  (f32 lane and prologue source)
  const int8_t* xq;       // i8 lane, PRO_X_F32 with pre-quantised input (may be null)
  const void* xd;         // f16 [K/32]
  const void* norm_w;
  float eps;
  int epi;               // GemvEpi; EPI_SWIGLU (ring form): y = f32 silu(gate) * up [R / 2]
  float* y;
  int w_evict_first;      // ring form: weight copies marked evict-first in L2
  int* claim;             // ring form: two zero ints; part of the rows is claimed by free CTAs
  int32_t* dots;          // i8 lane, EPI_STORE: also store the int32 block dots [R, K/32] the
                          // launch forms (test export of their bit-exactness); null: none
};
bool gemv_q8_supported(int K);
// True when a Q8_0 GEMV of K columns takes the ring form and can take EPI_SWIGLU.
bool gemv_q8_swiglu_ok(int K);
cudaError_t launch_gemv_q8(const GemvQ8Args& a, const Launch& L);
cudaError_t launch_quantize_q8(const float* x, int n, int8_t* xq, void* xd, const Launch& L);

// ----------------------------------------------------------------- attention
struct AttnArgs {
  // q source: either ready q (f32 [B, Hq, D]) or the fused QKV output
  const float* q;         // ready q, or null
  const float* qkv;       // f32 [B, (Hq + 2Hkv) * D] (fused mode), or null
  const void* q_norm;     // bf16 [D] (fused)
  const void* k_norm;     // bf16 [D] (fused)
  const float* rope;      // f32 [rope_max_pos, D/2, 2] (fused)
  int rope_max_pos;
  float eps;
  int act_bf16;           // fused: QK-norm output rounded to bf16 (bf16 activations)
  const int32_t* pos;     // fused: int32 [B], token position (keys 0..pos)
  const int32_t* seq_lens;// standalone: int32 [B], keys 0..len-1
  void* k_pages;          // bf16 [n_pages, Hkv, ps, D]
  void* v_pages;
  const int32_t* page_table;
  int B, Hq, Hkv, D, page_size, max_pages, n_pages;
  float scale;
  float* out_f32;         // standalone output f32 [B, Hq, D]
  void* out_bf16;         // fused output bf16 [B, Hq*D]
  void* workspace;
  size_t ws_bytes;
  int max_ctx;            // upper bound of keys per sequence (sizes the split grid)
  int use_cluster;        // fused form: > 1 splits each sequence over a cluster of at most this many CTAs
  L2Prefetch pf[2];       // CUDA-core form: weights of the GEMVs that follow, fetched into L2
                          // once the dependency wait is over (zero: none)
  int pf_late;            // 1: only once the CTA's own K/V tiles have all arrived
  const void* k_next;     // CUDA-core fused form: the next layer's caches (same shape);
  const void* v_next;     // each CTA fetches its split's cached rows of them into L2
  int kv_pf;              // 0 off, 1 evict-normal, 2 evict-last prefetch of k/v_next
  int trig_loop;          // CUDA-core form: let the next kernel launch only once this
                          // CTA's K/V loop is done (its weight prefetch then does not
                          // compete with the K/V tiles); 0: at the start
  int kv_ready;           // fused form: the current token's K/V rows are already in the
                          // cache (written by launch_kv_write); read them from there and
                          // do not write them (several rows of one sequence in one launch)
};
size_t attn_workspace_bytes(int B, int Hq, int Hkv, int max_ctx);
int attn_chunk(int B, int Hkv, int max_ctx);
cudaError_t launch_attention_mma(const AttnArgs& a, int chunk, size_t slots, const Launch& L);
cudaError_t launch_attention(const AttnArgs& a, const Launch& L);
// Static scratch of the allocation-free attention entry point: its capacity,
// and its device address with the ticket counters of the shape's workspace
// cleared on `stream` (no allocation).
size_t attn_noalloc_scratch_bytes();
cudaError_t attn_noalloc_scratch(int B, int Hq, int Hkv, int max_ctx, void** ptr, cudaStream_t stream);
cudaError_t launch_rope_table(float* table, int max_pos, int head_dim, float theta, cudaStream_t s);
// K/V rows of the current tokens into the cache: for row b < B and kv head g,
// k = RoPE_pos[b](RMSNorm(qkv[b] k-head g; k_norm)) and v, both rounded to bf16, at
// logical position pos[b] through page_table row b (the attention's fused prologue
// arithmetic, with bf16 activations when act_bf16).
// Row b's page table starts at page_table + b * pt_stride (0: all rows share one).
cudaError_t launch_kv_write(const float* qkv, int B, int Hq, int Hkv, const void* k_norm, const float* rope,
                            int rope_max_pos, float eps, int act_bf16, const int32_t* pos, const int32_t* page_table,
                            int pt_stride, int page_size, int max_pages, int n_pages, void* k_pages, void* v_pages,
                            const Launch& L);

// Speculative-verify attention (attention_verify.cu): the k rows of one sequence at
// positions pos[0..k) (their K/V already in the cache), q from qkv [k, QKV] with the
// QK-RMSNorm and RoPE fused in, every K/V tile read once for all k * Hq / Hkv query
// columns; page_table: the sequence's row. The workspace is the decode attention's for
// B = k rows.
bool verify_attention_supported(int k, int Hq, int Hkv);
cudaError_t launch_verify_attention(const AttnArgs& a, int k, const Launch& L);

// ----------------------------------------------------------------- prefill (prefill.cu)
// Causal attention of the n prompt rows of one sequence (positions pos[0] + i) over
// the cached keys 0 .. pos[0] + i, with the queries' QK-RMSNorm and RoPE fused in.
struct PrefillAttnArgs {
  const float* qkv;        // f32 [n, (Hq + 2 Hkv) D] (the QKV projection of the rows)
  int n, Hq, Hkv, D;       // D == 128
  const void* q_norm;      // bf16 [D]
  const float* rope;       // (cos, sin) table [rope_max_pos, D / 2]
  int rope_max_pos;
  float eps;
  int act_bf16;
  const int32_t* pos;      // pos[0]: position of row 0
  const void* k_pages;     // bf16 [n_pages, Hkv, page_size, D], the rows' K/V already written
  const void* v_pages;
  const int32_t* page_table;   // the sequence's page table [max_pages]
  int page_size, max_pages, n_pages;
  float scale;
  void* out;               // bf16 [n, Hq D]
};
cudaError_t launch_prefill_attention(const PrefillAttnArgs& a, const Launch& L);
// The tcgen05 form (prefill_tc.cu): a packing kernel copies the kv heads' keys [0, pos[0]
// + n) into `scratch` (K as is, V transposed; prefill_attention_tc_scratch_bytes bytes,
// cap = max_pages * page_size), then the attention reads them by TMA.
size_t prefill_attention_tc_scratch_bytes(int Hkv, int cap);
cudaError_t launch_prefill_attention_tc(const PrefillAttnArgs& a, void* scratch, size_t scratch_bytes,
                                        const Launch& L);
cudaError_t launch_prefill_prep(const int32_t* pos, int n, int32_t* vpos, const Launch& L);
cudaError_t launch_prefill_finish(int32_t* pos, int n, const Launch& L);

// ----------------------------------------------------------------- persistent batch-1 step
// The whole decode step of a BF16 model at batch 1 as one cooperative kernel
// (step_stream.cu). res / qkv / attn / h are the step workspace's activation
// buffers (f32 [H], f32 [QKV], bf16 [Hq D], bf16 [F]); ws is its own zero-filled
// scratch of stream_ws_bytes() (split partials, phase counters, argmax candidates),
// which every launch leaves zero-filled again unless a wait timed out.
constexpr int kStreamMaxLayers = 64;
struct StreamLayerPtrs {
  const void *w_qkv, *w_o, *w_gu, *w_down, *ln_in, *ln_post, *q_norm, *k_norm;
  void *k_cache, *v_cache;
};
struct StreamStepArgs {
  const StreamLayerPtrs* layers;  // host array [n_layers]
  int n_layers, H, Hq, Hkv, F, V;
  float eps;
  const void *embed, *final_norm, *lm_head;
  const int32_t* page_table;
  int page_size, max_pages, n_pages;
  const float* rope;
  int rope_max_pos;
  int32_t *tok, *pos, *step, *out_tokens;
  int max_steps;
  float* logits;
  float* res;
  float* qkv;
  void* attn;
  void* h;
  void* ws;
};
size_t stream_ws_bytes(int n_layers, int Hq, int Hkv);
bool stream_step_supported(const StreamStepArgs& a);
cudaError_t launch_stream_step(const StreamStepArgs& a, const Launch& L);

// ----------------------------------------------------------------- misc
size_t argmax_workspace_bytes(int B);
cudaError_t launch_argmax_advance(const float* logits, int V, int B, int32_t* tok, int32_t* pos,
                                  int32_t* step, int32_t* out_tokens, int max_steps, void* ws,
                                  const Launch& L);
cudaError_t launch_embed(const void* embed, int H, int V, const int32_t* tok, int B, float* res,
                         const Launch& L);
// Speculative verify (one sequence, k rows): row inputs tokens[i] = i ? draft[i - 1]
// : tok[0], positions pos[0] + i, page-table row 0 copied k times, and scratch
// argmax state zeroed; then, after the rows' argmax into target[k], the accepted
// prefix m (draft[i] == target[i] for i < m, m <= k - 1), out_tokens[step ..] =
// draft[0 .. m - 1], target[m]; tok = target[m], pos += m + 1, step += m + 1.
cudaError_t launch_verify_prep(const int32_t* tok, const int32_t* pos, const int32_t* draft, int k,
                               const int32_t* page_table, int max_pages, int32_t* tokens, int32_t* vpos,
                               int32_t* vpt, int32_t* scratch, const Launch& L);
// A bounded wait that runs out after limit_us (test of the timeout path).
cudaError_t launch_wait_timeout(int limit_us, const Launch& L);
cudaError_t launch_verify_accept(const int32_t* draft, const int32_t* target, int k, int32_t* tok, int32_t* pos,
                                 int32_t* step, int32_t* out_tokens, int max_steps, int32_t* n_accept,
                                 const Launch& L);
cudaError_t launch_paged_indices(const int32_t* pt, int B, int max_pages, int ps, int n_pages, int n_tokens,
                                 int32_t* idx, const Launch& L);

}  // namespace qd
