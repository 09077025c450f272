// C ABI of libqd.so: argument validation, the decode-step schedule and the
// whole-step CUDA graph. Kernels live in the other translation units.
//
// "GPU Kernel Lab" README, "Decode integration": the order of one decode step
// and its fixed-address CUDA graph replay. "emit_qwen38_generate" rustdoc,
// "Where the speed comes from": one launch per shared activation, one graph per
// token with token/position advanced on the device, residual + norm (+ Q8
// re-quantisation) fused into one kernel.
#include "qd.h"
#include "kernels.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

namespace qd {

static thread_local std::string g_last_error;

static int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
static int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

static int cuda_fail(cudaError_t e, const char* what) {
  cudaGetLastError();  // a rejected launch must not leave its error for the caller's next CUDA call
  return fail(QD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Sticky device error word; kernels receive its device address.
__device__ int g_dev_error = 0;

static int* dev_error_ptr() {
  static int* ptr[64] = {nullptr};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return nullptr;
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_error) != cudaSuccess) return nullptr;
    ptr[dev] = (int*)p;
  }
  return ptr[dev];
}

const DevInfo& dev_info() {
  static DevInfo info[64];
  static bool have[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!have[dev]) {
    cudaDeviceGetAttribute(&info[dev].sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&info[dev].max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (info[dev].sm_count <= 0) info[dev].sm_count = 1;
    have[dev] = true;
  }
  return info[dev];
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// QD_PDL=0 turns programmatic dependent launch off in the decode step (A/B timing).
static bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("QD_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

// By default a dependent kernel may launch as soon as this one starts (its
// CTAs take SMs as this kernel's CTAs finish and prefetch their weights);
// QD_PDL_TRIGGER=late holds it until this kernel has issued its last weight /
// KV copy. Both measured within 0.5% of each other on the Qwen3-8B step.
static int pdl_trigger_late() {
  static const int late = [] {
    const char* v = getenv("QD_PDL_TRIGGER");
    return (v && strcmp(v, "late") == 0) ? 1 : 0;
  }();
  return late;
}

// QD_ATTN_CLUSTER=n (2..16) makes the decode step split each sequence over a
// thread block cluster of at most n CTAs; the default (0) uses the workspace
// split-KV form, which measured faster on the Qwen3-8B step.
static int attn_cluster_enabled() {
  static const int n = [] {
    const char* v = getenv("QD_ATTN_CLUSTER");
    return v ? atoi(v) : 0;
  }();
  return n;
}

// L2 prefetch of weights ahead of the GEMV that reads them (batch-1 BF16 step):
// QD_L2PF_ATTN_WO_KB = leading KB of every O-projection span that the attention
// kernel fetches (QD_L2PF_ATTN_LATE = 1: after its own K/V, else right after
// the dependency wait);
// QD_L2PF_ATTN_GU_KB = leading KB of every gate+up span it fetches as well;
// QD_L2PF_TAIL_KB = leading KB of every span of the next GEMV that a ring GEMV
// fetches once its own copies are issued. 0 turns a form off. Defaults (64 KB of
// O-projection spans after the attention's K/V, 96 KB tails): 335.1 vs 329.1 tok/s
// on the Qwen3-8B step, same box; whole-matrix or early prefetches were slower.
// QD_ATTN_TRIGGER_LOOP = 1: the attention lets the O projection launch only once
// its K/V loop is done. QD_GEMV_O_RING_KB: ring size of the O projection.
// QD_SWIGLU_IN_DOWN = 1: form SwiGLU in the down projection's prologue instead of
// the gate+up epilogue (batch 1).
// QD_KV_PF = 1 / 2: each attention fetches its split's rows of the next layer's
// caches into L2 (evict-normal / evict-last; measured no gain on the Qwen3-8B
// step). QD_W_EVICT_FIRST (default 1) marks GEMV weight copies evict-first in L2,
// so the streamed weights do not push activations and caches out (measured
// 1.7 % faster on the Qwen3-8B step).
// QD_GEMV_DOWN_RING_KB / QD_GEMV_QKV_RING_KB: ring size of the down / QKV projection.
struct StepTuning {
  int down_ring_kb = 0;
  int qkv_ring_kb = 0;
  int kv_pf = 0;
  int w_evict_first = 1;
  int swiglu_in_down = 0;
  int attn_trig_loop = 0;
  int o_ring_kb = 0;
  long long attn_wo_kb = 64;   // measured best with the two below on the Qwen3-8B step
  int attn_late = 1;
  long long attn_gu_kb = 0;
  long long tail_kb = 96;
};
static const StepTuning& step_tuning() {
  static const StepTuning t = [] {
    StepTuning u;
    if (const char* v = getenv("QD_L2PF_ATTN_WO_KB")) u.attn_wo_kb = std::max(0LL, atoll(v));
    if (const char* v = getenv("QD_L2PF_ATTN_LATE")) u.attn_late = atoi(v) != 0;
    if (const char* v = getenv("QD_L2PF_ATTN_GU_KB")) u.attn_gu_kb = std::max(0LL, atoll(v));
    if (const char* v = getenv("QD_L2PF_TAIL_KB")) u.tail_kb = std::max(0LL, atoll(v));
    if (const char* v = getenv("QD_ATTN_TRIGGER_LOOP")) u.attn_trig_loop = atoi(v) != 0;
    if (const char* v = getenv("QD_SWIGLU_IN_DOWN")) u.swiglu_in_down = atoi(v) != 0;
    if (const char* v = getenv("QD_KV_PF")) u.kv_pf = std::max(0, std::min(2, atoi(v)));
    if (const char* v = getenv("QD_GEMV_DOWN_RING_KB")) u.down_ring_kb = std::max(0, atoi(v));
    if (const char* v = getenv("QD_GEMV_QKV_RING_KB")) u.qkv_ring_kb = std::max(0, atoi(v));
    if (const char* v = getenv("QD_W_EVICT_FIRST")) u.w_evict_first = atoi(v) != 0;
    if (const char* v = getenv("QD_GEMV_O_RING_KB")) u.o_ring_kb = std::max(0, atoi(v));
    return u;
  }();
  return t;
}

// Small-batch BF16 implementation, QD_SMALLB_IMPL (read per call): "mma" (default) runs
// batch 2..8 on the mma.sync weight-streaming GEMV; "tc" on the tcgen05 GEMMs from
// QD_TC_MIN_BATCH; "simt" on the CUDA-core GEMV up to batch 8.
enum { SMALLB_MMA = 0, SMALLB_TC = 1, SMALLB_SIMT = 2 };
static int small_batch_impl() {
  const char* e = getenv("QD_SMALLB_IMPL");
  if (e && strcmp(e, "tc") == 0) return SMALLB_TC;
  if (e && strcmp(e, "simt") == 0) return SMALLB_SIMT;
  return SMALLB_MMA;
}

// Small-batch GEMVs, QD_MMA_NORM_ROWS (read per call): 1 (default) runs each RMSNorm
// as a row kernel writing the bf16 rows once, 0 in every GEMV CTA's prologue. The row
// kernel measured faster on the Qwen3-8B step: 609 / 1135 / 1790 against
// 524 / 997 / 1606 tok/s at batch 2 / 4 / 8 (each prologue re-read the f32 rows
// before its first MMA).
static bool mma_norm_rows() {
  const char* v = getenv("QD_MMA_NORM_ROWS");
  return v == nullptr || atoi(v) != 0;
}

static Launch make_launch(cudaStream_t s, bool pdl) {
  Launch L;
  L.stream = s;
  L.trig_late = pdl_trigger_late();
  L.pdl = pdl && pdl_enabled();
  L.err = dev_error_ptr();
  return L;
}

}  // namespace qd

using namespace qd;

struct qd_layer {
  qd_layer_dims dims;
  qd_layer_weights w;
};

struct qd_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  int steps;
};

extern "C" {

const char* qd_last_error(void) { return qd::g_last_error.c_str(); }
int qd_version(void) { return 1; }

// ------------------------------------------------------------------ GEMVs
int qd_gemv_bf16(const void* W, int rows, int cols, const void* x, int x_is_f32, float* y, int batch,
                 cudaStream_t stream) {
  if (!W || !x || !y) return fail(QD_ERR_INVALID_ARG, "qd_gemv_bf16: null pointer");
  if (rows < 1 || cols < 8) return fail(QD_ERR_INVALID_ARG, "qd_gemv_bf16: rows=%d cols=%d", rows, cols);
  if (!aligned16(W) || !aligned16(x) || !aligned16(y))
    return fail(QD_ERR_INVALID_ARG, "qd_gemv_bf16: pointers must be 16-byte aligned");
  if (batch > 8) {  // a real contraction: tcgen05 tensor cores
    const bool ok = batch <= 64 ? gemm_tc_supported(rows, cols, batch) : gemm_tc_rows_supported(rows, cols, batch, false);
    if (x_is_f32 || !ok)
      return fail(QD_ERR_UNSUPPORTED, "qd_gemv_bf16: batch %d needs bf16 x and cols %% 64 == 0", batch);
    GemmTcArgs g = {};
    g.W = W; g.X = x; g.R = rows; g.K = cols; g.B = batch; g.epi = EPI_STORE; g.y = y;
    cudaError_t e = launch_gemm_tc(g, make_launch(stream, false));
    return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_gemv_bf16 (tensor cores)");
  }
  if (batch >= 2 && !x_is_f32 && small_batch_impl() == SMALLB_MMA && gemv_mma_supported(rows, cols, batch)) {
    GemvMmaArgs g = {};
    g.W = W; g.R = rows; g.K = cols; g.B = batch; g.pro = PRO_X_BF16; g.x = x; g.epi = EPI_STORE; g.y = y;
    g.w_evict_first = 1;
    cudaError_t e = launch_gemv_mma(g, make_launch(stream, false));
    return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_gemv_bf16 (mma.sync)");
  }
  if (!gemv_bf16_supported(cols, batch))
    return fail(QD_ERR_UNSUPPORTED, "qd_gemv_bf16: cols=%d batch=%d (need cols%%8==0, cols<=32768, 1<=batch<=8)",
                cols, batch);
  GemvBf16Args a = {};
  a.W = W; a.R = rows; a.K = cols; a.batch = batch;
  a.pro = x_is_f32 ? PRO_X_F32 : PRO_X_BF16;
  a.x = x; a.norm_w = nullptr; a.eps = 0.f;
  a.epi = EPI_STORE; a.y = y;
  cudaError_t e = launch_gemv_bf16(a, make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_gemv_bf16");
}

int qd_gemv_q8_0(const int8_t* qs, const void* d_f16, int rows, int cols, const float* x_f32,
                 const int8_t* x_q, const void* x_d_f16, qd_act act, float* y, cudaStream_t stream) {
  if (!qs || !d_f16 || !y) return fail(QD_ERR_INVALID_ARG, "qd_gemv_q8_0: null pointer");
  if (rows < 1 || cols < 32 || cols % 32) return fail(QD_ERR_INVALID_ARG, "qd_gemv_q8_0: rows=%d cols=%d", rows, cols);
  if (!gemv_q8_supported(cols)) return fail(QD_ERR_UNSUPPORTED, "qd_gemv_q8_0: cols=%d too large", cols);
  if (act == QD_ACT_F32 && !x_f32) return fail(QD_ERR_INVALID_ARG, "qd_gemv_q8_0: f32 lane needs x_f32");
  if (act == QD_ACT_I8 && !(x_q && x_d_f16) && !x_f32)
    return fail(QD_ERR_INVALID_ARG, "qd_gemv_q8_0: i8 lane needs x_q and x_d (or x_f32 to quantise)");
  if (act != QD_ACT_F32 && act != QD_ACT_I8) return fail(QD_ERR_INVALID_ARG, "qd_gemv_q8_0: bad act");
  if (!aligned16(qs) || !aligned16(y) || (x_f32 && !aligned16(x_f32)) || (x_q && !aligned16(x_q)))
    return fail(QD_ERR_INVALID_ARG, "qd_gemv_q8_0: pointers must be 16-byte aligned");
  if (((uintptr_t)d_f16 & 1u) || (x_d_f16 && ((uintptr_t)x_d_f16 & 1u)))
    return fail(QD_ERR_INVALID_ARG, "qd_gemv_q8_0: scale pointers must be 2-byte aligned");
  GemvQ8Args a = {};
  a.qs = qs; a.d = d_f16; a.R = rows; a.K = cols; a.act = act;
  a.pro = PRO_X_F32; a.x = x_f32;
  a.xq = (act == QD_ACT_I8 && x_q && x_d_f16) ? x_q : nullptr; a.xd = x_d_f16;
  a.norm_w = nullptr; a.eps = 0.f; a.epi = EPI_STORE; a.y = y;
  cudaError_t e = launch_gemv_q8(a, make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_gemv_q8_0");
}

size_t qd_gemv_w4_workspace_bytes(int rows, int cols) {
  if (rows < 1 || !gemv_w4_tc_supported(cols)) return 0;
  return gemv_w4_tc_workspace_bytes(rows, cols, false);
}

int qd_gemv_w4_ex(const uint8_t* W, const void* d_f16, int rows, int cols, const void* x_bf16, float* y,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!W || !d_f16 || !x_bf16 || !y) return fail(QD_ERR_INVALID_ARG, "qd_gemv_w4: null pointer");
  if (rows < 1 || !gemv_w4_supported(cols))
    return fail(QD_ERR_INVALID_ARG, "qd_gemv_w4: rows=%d cols=%d (cols %% 32 == 0, <= 16384)", rows, cols);
  if (!aligned16(W) || !aligned16(x_bf16) || !aligned16(y) || ((uintptr_t)d_f16 & 1u) ||
      (workspace && !aligned16(workspace)))
    return fail(QD_ERR_INVALID_ARG, "qd_gemv_w4: alignment");
  GemvW4Args g = {};
  g.W = W; g.d = d_f16; g.R = rows; g.K = cols; g.pro = PRO_X_BF16; g.x = x_bf16; g.epi = EPI_STORE; g.y = y;
  g.split_ws = workspace; g.split_ws_bytes = workspace ? workspace_bytes : 0;
  cudaError_t e = launch_gemv_w4(g, make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_gemv_w4");
}

int qd_gemv_w4(const uint8_t* W, const void* d_f16, int rows, int cols, const void* x_bf16, float* y,
               cudaStream_t stream) {
  return qd_gemv_w4_ex(W, d_f16, rows, cols, x_bf16, y, nullptr, 0, stream);
}

size_t qd_w4_topk_workspace_bytes(void) { return w4_topk_workspace_bytes(); }

int qd_gemv_w4_topk(const uint8_t* W, const void* d_f16, int rows, int cols, const void* x_bf16, int k, float* y,
                    int32_t* topk_ids, float* topk_vals, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream) {
  if (!W || !d_f16 || !x_bf16 || !y || !topk_ids || !topk_vals || !workspace)
    return fail(QD_ERR_INVALID_ARG, "qd_gemv_w4_topk: null pointer");
  if (rows < 1 || !gemv_w4_supported(cols) || k < 1 || k > 16)
    return fail(QD_ERR_INVALID_ARG, "qd_gemv_w4_topk: rows=%d cols=%d k=%d", rows, cols, k);
  if (!aligned16(W) || !aligned16(x_bf16) || !aligned16(y) || !aligned16(workspace) || ((uintptr_t)d_f16 & 1u))
    return fail(QD_ERR_INVALID_ARG, "qd_gemv_w4_topk: alignment");
  if (workspace_bytes < w4_topk_workspace_bytes()) return fail(QD_ERR_WORKSPACE, "qd_gemv_w4_topk: workspace");
  GemvW4Args g = {};
  g.W = W; g.d = d_f16; g.R = rows; g.K = cols; g.pro = PRO_X_BF16; g.x = x_bf16; g.epi = EPI_TOPK; g.y = y;
  g.top_k = k; g.ws = workspace; g.topk_ids = topk_ids; g.topk_vals = topk_vals;
  cudaError_t e = launch_gemv_w4(g, make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_gemv_w4_topk");
}

size_t qd_gemm_workspace_bytes(int rows, int cols, qd_wtype wtype) {
  if (rows < 1 || cols < 1) return 0;
  return gemm_tc_workspace_bytes(rows, cols, wtype == QD_W_Q8_0);
}

int qd_gemm_q8_0(const int8_t* qs, const void* d_f16, int rows, int cols, const void* x_bf16, int batch, float* y,
                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!qs || !d_f16 || !x_bf16 || !y) return fail(QD_ERR_INVALID_ARG, "qd_gemm_q8_0: null pointer");
  if (rows < 1 || cols < 32 || cols % 32 || batch < 1)
    return fail(QD_ERR_INVALID_ARG, "qd_gemm_q8_0: rows=%d cols=%d batch=%d", rows, cols, batch);
  if (batch <= 64 ? !gemm_tc_q8_supported(rows, cols, batch) : !gemm_tc_rows_supported(rows, cols, batch, true))
    return fail(QD_ERR_UNSUPPORTED, "qd_gemm_q8_0: need cols %% 256 == 0 (cols=%d batch=%d)", cols, batch);
  if (!aligned16(qs) || !aligned16(d_f16) || !aligned16(x_bf16) || !aligned16(y) ||
      (workspace && !aligned16(workspace)))
    return fail(QD_ERR_INVALID_ARG, "qd_gemm_q8_0: pointers must be 16-byte aligned");
  GemmTcArgs g = {};
  g.W = qs; g.S = d_f16; g.X = x_bf16; g.R = rows; g.K = cols; g.B = batch; g.epi = EPI_STORE; g.y = y;
  g.ws = workspace; g.ws_bytes = workspace ? workspace_bytes : 0;
  cudaError_t e = launch_gemm_tc(g, make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_gemm_q8_0");
}

int qd_quantize_q8_0(const float* x, int n, int8_t* x_q, void* x_d_f16, cudaStream_t stream) {
  if (!x || !x_q || !x_d_f16) return fail(QD_ERR_INVALID_ARG, "qd_quantize_q8_0: null pointer");
  if (n < 0 || n % 32) return fail(QD_ERR_INVALID_ARG, "qd_quantize_q8_0: n=%d must be a multiple of 32", n);
  if (n == 0) return QD_OK;
  cudaError_t e = launch_quantize_q8(x, n, x_q, x_d_f16, make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_quantize_q8_0");
}

// ------------------------------------------------------------------ attention
size_t qd_attn_workspace_bytes(int batch, int n_q_heads, int n_kv_heads, int max_ctx) {
  if (batch < 1 || n_kv_heads < 1 || n_q_heads < n_kv_heads || max_ctx < 1) return 0;
  return attn_workspace_bytes(batch, n_q_heads, n_kv_heads, max_ctx);
}

static int check_attn_shape(const char* fn, int batch, int hq, int hkv, int hd, int ps, int max_pages,
                            int n_pages) {
  if (batch < 1 || hq < 1 || hkv < 1 || ps < 1 || max_pages < 1 || n_pages < 1)
    return fail(QD_ERR_INVALID_ARG, "%s: bad sizes batch=%d hq=%d hkv=%d page_size=%d max_pages=%d n_pages=%d", fn,
                batch, hq, hkv, ps, max_pages, n_pages);
  if (hd != 128) return fail(QD_ERR_UNSUPPORTED, "%s: head_dim=%d (only 128)", fn, hd);
  if (hq % hkv) return fail(QD_ERR_INVALID_ARG, "%s: n_q_heads %% n_kv_heads != 0", fn);
  const int rep = hq / hkv;
  if (rep != 1 && rep != 2 && rep != 4 && rep != 8)
    return fail(QD_ERR_UNSUPPORTED, "%s: n_q_heads/n_kv_heads=%d (supported 1, 2, 4, 8)", fn, rep);
  if ((long long)max_pages * ps > (1LL << 30)) return fail(QD_ERR_INVALID_ARG, "%s: context too large", fn);
  return QD_OK;
}

int qd_attn_decode_paged(const float* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                         const int32_t* seq_lens, int batch, int n_q_heads, int n_kv_heads, int head_dim,
                         int page_size, int max_pages, int n_pages, float scale, float* out, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_attn_shape("qd_attn_decode_paged", batch, n_q_heads, n_kv_heads, head_dim, page_size, max_pages,
                            n_pages);
  if (rc) return rc;
  if (!q || !k_pages || !v_pages || !page_table || !seq_lens || !out || !workspace)
    return fail(QD_ERR_INVALID_ARG, "qd_attn_decode_paged: null pointer");
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out) || !aligned16(workspace))
    return fail(QD_ERR_INVALID_ARG, "qd_attn_decode_paged: pointers must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(QD_ERR_INVALID_ARG, "qd_attn_decode_paged: scale not finite");
  const int max_ctx = max_pages * page_size;
  const size_t need = attn_workspace_bytes(batch, n_q_heads, n_kv_heads, max_ctx);
  if (workspace_bytes < need)
    return fail(QD_ERR_WORKSPACE, "qd_attn_decode_paged: workspace %zu < %zu bytes", workspace_bytes, need);
  AttnArgs a = {};
  a.q = q; a.seq_lens = seq_lens;
  a.k_pages = (void*)k_pages; a.v_pages = (void*)v_pages; a.page_table = page_table;
  a.B = batch; a.Hq = n_q_heads; a.Hkv = n_kv_heads; a.D = head_dim;
  a.page_size = page_size; a.max_pages = max_pages; a.n_pages = n_pages;
  a.scale = scale; a.out_f32 = out; a.workspace = workspace; a.ws_bytes = workspace_bytes; a.max_ctx = max_ctx;
  cudaError_t e = launch_attention(a, make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_attn_decode_paged");
}

int qd_attn_decode_paged_noalloc(const float* q, const void* k_pages, const void* v_pages,
                                 const int32_t* page_table, const int32_t* seq_lens, int batch, int n_q_heads,
                                 int n_kv_heads, int head_dim, int page_size, int max_pages, int n_pages,
                                 float scale, float* out, cudaStream_t stream) {
  int rc = check_attn_shape("qd_attn_decode_paged_noalloc", batch, n_q_heads, n_kv_heads, head_dim, page_size,
                            max_pages, n_pages);
  if (rc) return rc;
  if (!q || !k_pages || !v_pages || !page_table || !seq_lens || !out)
    return fail(QD_ERR_INVALID_ARG, "qd_attn_decode_paged_noalloc: null pointer");
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
    return fail(QD_ERR_INVALID_ARG, "qd_attn_decode_paged_noalloc: pointers must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(QD_ERR_INVALID_ARG, "qd_attn_decode_paged_noalloc: scale not finite");
  const int max_ctx = max_pages * page_size;
  const size_t need = attn_workspace_bytes(batch, n_q_heads, n_kv_heads, max_ctx);
  if (need > attn_noalloc_scratch_bytes())
    return fail(QD_ERR_WORKSPACE,
                "qd_attn_decode_paged_noalloc: this shape needs %zu bytes of scratch, more than the %zu-byte "
                "static array; use qd_attn_decode_paged with a caller-provided workspace",
                need, attn_noalloc_scratch_bytes());
  void* scratch = nullptr;
  cudaError_t e = attn_noalloc_scratch(batch, n_q_heads, n_kv_heads, max_ctx, &scratch, stream);
  if (e != cudaSuccess) return cuda_fail(e, "qd_attn_decode_paged_noalloc: scratch set-up");
  AttnArgs a = {};
  a.q = q; a.seq_lens = seq_lens;
  a.k_pages = (void*)k_pages; a.v_pages = (void*)v_pages; a.page_table = page_table;
  a.B = batch; a.Hq = n_q_heads; a.Hkv = n_kv_heads; a.D = head_dim;
  a.page_size = page_size; a.max_pages = max_pages; a.n_pages = n_pages;
  a.scale = scale; a.out_f32 = out; a.workspace = scratch; a.ws_bytes = need; a.max_ctx = max_ctx;
  e = launch_attention(a, make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_attn_decode_paged_noalloc");
}

// ------------------------------------------------------------------ argmax
size_t qd_argmax_workspace_bytes(int batch) { return batch < 1 ? 0 : argmax_workspace_bytes(batch); }

int qd_argmax_advance(const float* logits, int vocab, int batch, int32_t* tok, int32_t* pos, int32_t* step,
                      int32_t* out_tokens, int max_steps, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  if (!logits || !tok || !pos || !step || !out_tokens || !workspace)
    return fail(QD_ERR_INVALID_ARG, "qd_argmax_advance: null pointer");
  if (vocab < 1 || batch < 1 || max_steps < 1)
    return fail(QD_ERR_INVALID_ARG, "qd_argmax_advance: vocab=%d batch=%d max_steps=%d", vocab, batch, max_steps);
  if (workspace_bytes < argmax_workspace_bytes(batch))
    return fail(QD_ERR_WORKSPACE, "qd_argmax_advance: workspace too small");
  cudaError_t e = launch_argmax_advance(logits, vocab, batch, tok, pos, step, out_tokens, max_steps, workspace,
                                        make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_argmax_advance");
}

int qd_rope_table_init(float* table, int max_pos, int head_dim, float theta, cudaStream_t stream) {
  if (!table || max_pos < 1 || head_dim < 2 || head_dim % 2 || !(theta > 0.f))
    return fail(QD_ERR_INVALID_ARG, "qd_rope_table_init: bad arguments");
  cudaError_t e = launch_rope_table(table, max_pos, head_dim, theta, stream);
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_rope_table_init");
}

// ------------------------------------------------------------------ layers
int qd_create_layer(const qd_layer_dims* d, const qd_layer_weights* w, qd_layer** out) {
  if (!d || !w || !out) return fail(QD_ERR_INVALID_ARG, "qd_create_layer: null pointer");
  *out = nullptr;
  if (d->hidden < 32 || d->ffn < 32 || d->n_q_heads < 1 || d->n_kv_heads < 1)
    return fail(QD_ERR_INVALID_ARG, "qd_create_layer: bad dims");
  if (d->head_dim != 128) return fail(QD_ERR_UNSUPPORTED, "qd_create_layer: head_dim=%d (only 128)", d->head_dim);
  if (d->n_q_heads % d->n_kv_heads) return fail(QD_ERR_INVALID_ARG, "qd_create_layer: Hq %% Hkv != 0");
  const int rep = d->n_q_heads / d->n_kv_heads;
  if (rep != 1 && rep != 2 && rep != 4 && rep != 8) return fail(QD_ERR_UNSUPPORTED, "qd_create_layer: Hq/Hkv=%d", rep);
  if (!(d->rms_eps >= 0.f) || !(d->rope_theta > 0.f)) return fail(QD_ERR_INVALID_ARG, "qd_create_layer: eps/theta");
  if (!w->w_qkv || !w->w_o || !w->w_gu || !w->w_down || !w->ln_in || !w->ln_post || !w->q_norm || !w->k_norm)
    return fail(QD_ERR_INVALID_ARG, "qd_create_layer: null weight pointer");
  const int qdim = d->n_q_heads * d->head_dim;
  if (d->wtype == QD_W_BF16) {
    if (d->hidden % 8 || d->ffn % 8 || !gemv_bf16_supported(d->hidden, 1) || !gemv_bf16_supported(d->ffn, 1) ||
        !gemv_bf16_supported(qdim, 1))
      return fail(QD_ERR_UNSUPPORTED, "qd_create_layer: bf16 dims not supported");
  } else if (d->wtype == QD_W_INT4) {
    if (!gemv_w4_supported(d->hidden) || !gemv_w4_supported(d->ffn) || !gemv_w4_supported(qdim))
      return fail(QD_ERR_UNSUPPORTED, "qd_create_layer: INT4 dims need multiples of 32 up to 16384");
    if (!w->s_qkv || !w->s_o || !w->s_gu || !w->s_down)
      return fail(QD_ERR_INVALID_ARG, "qd_create_layer: INT4 scales missing");
  } else if (d->wtype == QD_W_Q8_0) {
    if (d->hidden % 32 || d->ffn % 32 || !gemv_q8_supported(d->hidden) || !gemv_q8_supported(d->ffn) ||
        !gemv_q8_supported(qdim))
      return fail(QD_ERR_UNSUPPORTED, "qd_create_layer: Q8_0 dims need multiples of 32");
    if (!w->s_qkv || !w->s_o || !w->s_gu || !w->s_down)
      return fail(QD_ERR_INVALID_ARG, "qd_create_layer: Q8_0 scales missing");
    if (d->act != QD_ACT_F32 && d->act != QD_ACT_I8) return fail(QD_ERR_INVALID_ARG, "qd_create_layer: bad act");
  } else {
    return fail(QD_ERR_INVALID_ARG, "qd_create_layer: bad wtype");
  }
  const void* ptrs[] = {w->w_qkv, w->w_o, w->w_gu, w->w_down, w->ln_in, w->ln_post, w->q_norm, w->k_norm};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(QD_ERR_INVALID_ARG, "qd_create_layer: weights must be 16-byte aligned");
  qd_layer* l = new qd_layer;
  l->dims = *d;
  l->w = *w;
  *out = l;
  return QD_OK;
}

int qd_destroy_layer(qd_layer* layer) {
  delete layer;
  return QD_OK;
}

// ------------------------------------------------------------------ decode step
namespace {

struct StepWs {
  float* res;       // [B, H]
  float* qkv;       // [B, QKV]
  void* attn;       // [B, Hq*D] bf16 or f32
  float* gu;        // [B, 2F]
  void* xn;         // bf16 [B, max(H, F)]: normed / SwiGLU activations (batched path)
  void* attn_ws;
  void* argmax_ws;
  int* claims;      // [5 L + 1][2] row-claim counters of the batch-1 Q8_0 GEMVs (zero between launches)
  void* gemm_ws;    // batched path: split-K partials and tickets (one GEMM at a time)
  size_t gemm_ws_bytes;
  void* stream_ws;  // batch-1 BF16: the persistent step kernel's partials, counters, candidates
  void* topk_ws;    // INT4 LM head: top-k candidates and ticket
  void* w4_ws;      // INT4 layers: split-K partials and tickets of the tcgen05 GEMVs (one at a time)
  size_t w4_ws_bytes;
  size_t total;
};

// The LM head's format: INT4 (lm_wtype), else Q8_0 when scales are given, else bf16.
bool lm_is_w4(const qd_step_args* a) { return a->lm_wtype == QD_W_INT4; }
bool lm_is_q8(const qd_step_args* a) { return a->lm_head_scales != nullptr && !lm_is_w4(a); }

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

// The mma.sync step: BF16 layers and LM head at batch 2..8 with every K a multiple
// of 32. Each projection streams its weights once for all rows at the batch-1
// GEMV's rate, with the RMSNorm in the prologue and SwiGLU in the gate+up epilogue.
bool mma_step(const qd_step_args* a) {
  const qd_layer_dims& d = a->layers[0]->dims;
  const int B = a->batch;
  return d.wtype == QD_W_BF16 && !a->lm_head_scales && B >= 2 && B <= 8 && small_batch_impl() == SMALLB_MMA &&
         gemv_mma_supported(1, d.hidden, B) && gemv_mma_supported(1, d.n_q_heads * d.head_dim, B) &&
         gemv_mma_supported(1, d.ffn, B);
}

// The tcgen05 step: BF16 models from batch 9 (from QD_TC_MIN_BATCH, default 3, when
// the small-batch implementation is "tc", or where the mma.sync step does not apply),
// Q8_0 models from batch 2 (the Q8_0 GEMV lanes take one activation vector). The
// batch 2..8 CUDA-core GEMV streams 3.84 / 2.67 / 0.96 TB/s at batch 2 / 4 / 8
// against ~3.9 for the tcgen05 GEMM, and its K limit rejects the 12288-wide down
// projection above batch 2.
bool tc_step(const qd_step_args* a) {
  static const int min_b = [] {
    const char* v = getenv("QD_TC_MIN_BATCH");
    return v ? std::max(2, atoi(v)) : 3;
  }();
  const qd_layer_dims& d = a->layers[0]->dims;
  if (d.wtype == QD_W_Q8_0) return a->batch > 1;
  if (a->batch > 8) return true;
  if (mma_step(a) || small_batch_impl() == SMALLB_SIMT) return false;
  // batch min_b .. 8: the tensor cores where their K rule holds, else the GEMV
  return a->batch >= min_b && d.hidden % 64 == 0 && (d.n_q_heads * d.head_dim) % 64 == 0 && d.ffn % 64 == 0;
}

StepWs step_ws_layout_for(const qd_step_args* a, void* base, bool gemm_path);
StepWs step_ws_layout(const qd_step_args* a, void* base) { return step_ws_layout_for(a, base, tc_step(a)); }
// gemm_path: size the split-K GEMM workspace (the step runs its projections as GEMMs)
StepWs step_ws_layout_for(const qd_step_args* a, void* base, bool gemm_path) {
  const qd_layer_dims& d = a->layers[0]->dims;
  const int B = a->batch;
  const size_t qkv = (size_t)(d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim;
  unsigned char* p = (unsigned char*)base;
  StepWs w;
  size_t off = 0;
  w.res = (float*)(p + off); off += al256((size_t)B * d.hidden * 4);
  w.qkv = (float*)(p + off); off += al256((size_t)B * qkv * 4);
  w.attn = (void*)(p + off); off += al256((size_t)B * d.n_q_heads * d.head_dim * 4);
  w.gu = (float*)(p + off); off += al256((size_t)B * 2 * d.ffn * 4);
  w.xn = (void*)(p + off); off += al256((size_t)B * std::max(d.hidden, d.ffn) * 2);
  w.attn_ws = (void*)(p + off);
  off += al256(attn_workspace_bytes(B, d.n_q_heads, d.n_kv_heads, a->max_pages * a->page_size));
  w.argmax_ws = (void*)(p + off); off += al256(argmax_workspace_bytes(B));
  w.claims = (int*)(p + off); off += al256((size_t)(5 * a->n_layers + 1) * 2 * sizeof(int));
  w.gemm_ws = (void*)(p + off);
  w.gemm_ws_bytes = 0;
  if (gemm_path) {  // the batched step runs its projections as split-K tcgen05 GEMMs
    const bool q8 = d.wtype == QD_W_Q8_0, q8_head = lm_is_q8(a);
    const int shapes[5][3] = {{(int)qkv, d.hidden, q8}, {d.hidden, d.n_q_heads * d.head_dim, q8},
                              {2 * d.ffn, d.hidden, q8}, {d.hidden, d.ffn, q8}, {a->vocab, d.hidden, q8_head}};
    for (const auto& sh : shapes)
      w.gemm_ws_bytes = std::max(w.gemm_ws_bytes, gemm_tc_workspace_bytes(sh[0], sh[1], sh[2] != 0));
  }
  off += al256(w.gemm_ws_bytes);
  w.stream_ws = (void*)(p + off);
  if (a->batch == 1 && d.wtype == QD_W_BF16) off += al256(stream_ws_bytes(a->n_layers, d.n_q_heads, d.n_kv_heads));
  w.topk_ws = (void*)(p + off);
  if (lm_is_w4(a)) off += al256(w4_topk_workspace_bytes());
  w.w4_ws = (void*)(p + off);
  w.w4_ws_bytes = 0;
  if (d.wtype == QD_W_INT4) {
    const int shapes[4][3] = {{(int)qkv, d.hidden, 0}, {d.hidden, d.n_q_heads * d.head_dim, 0},
                              {2 * d.ffn, d.hidden, 1}, {d.hidden, d.ffn, 0}};
    for (const auto& sh : shapes)
      w.w4_ws_bytes = std::max(w.w4_ws_bytes, gemv_w4_tc_workspace_bytes(sh[0], sh[1], sh[2] != 0));
  }
  off += al256(w.w4_ws_bytes);
  w.total = off;
  return w;
}

// QD_STEP_PATH (read on every call): "persistent" runs a batch-1 BF16 step as the
// one persistent step kernel (step_stream.cu) when its shape allows; anything else
// keeps the one-kernel-per-operation path.
bool step_kernels_forced() {
  const char* v = getenv("QD_STEP_PATH");
  return !(v && strcmp(v, "persistent") == 0);
}

// The persistent batch-1 step (step_stream.cu): its arguments, and whether it takes
// this step.
bool stream_args(const qd_step_args* a, const StepWs& w, std::vector<StreamLayerPtrs>& lp, StreamStepArgs& s) {
  const qd_layer_dims& d = a->layers[0]->dims;
  if (a->batch != 1 || d.wtype != QD_W_BF16 || a->lm_head_scales || a->n_layers > kStreamMaxLayers) return false;
  lp.resize(a->n_layers);
  for (int i = 0; i < a->n_layers; ++i) {
    const qd_layer_weights& lw = a->layers[i]->w;
    lp[i] = StreamLayerPtrs{lw.w_qkv, lw.w_o, lw.w_gu, lw.w_down, lw.ln_in, lw.ln_post, lw.q_norm, lw.k_norm,
                            a->k_cache[i], a->v_cache[i]};
  }
  s = StreamStepArgs{};
  s.layers = lp.data();
  s.n_layers = a->n_layers;
  s.H = d.hidden; s.Hq = d.n_q_heads; s.Hkv = d.n_kv_heads; s.F = d.ffn; s.V = a->vocab;
  s.eps = d.rms_eps;
  s.embed = a->embed; s.final_norm = a->final_norm; s.lm_head = a->lm_head;
  s.page_table = a->page_table; s.page_size = a->page_size; s.max_pages = a->max_pages; s.n_pages = a->n_pages;
  s.rope = a->rope_table; s.rope_max_pos = a->rope_max_pos;
  s.tok = a->tok; s.pos = a->pos; s.step = a->step; s.out_tokens = a->out_tokens; s.max_steps = a->max_steps;
  s.logits = a->logits;
  s.res = w.res; s.qkv = w.qkv; s.attn = w.attn; s.h = w.xn;
  s.ws = w.stream_ws;
  return stream_step_supported(s);
}

int validate_step(const qd_step_args* a) {
  if (!a) return fail(QD_ERR_INVALID_ARG, "qd_decode_step: null args");
  if (!a->layers || a->n_layers < 1) return fail(QD_ERR_INVALID_ARG, "qd_decode_step: no layers");
  for (int i = 0; i < a->n_layers; ++i)
    if (!a->layers[i]) return fail(QD_ERR_INVALID_ARG, "qd_decode_step: layer %d is null", i);
  const qd_layer_dims& d0 = a->layers[0]->dims;
  for (int i = 1; i < a->n_layers; ++i) {
    const qd_layer_dims& d = a->layers[i]->dims;
    if (d.hidden != d0.hidden || d.n_q_heads != d0.n_q_heads || d.n_kv_heads != d0.n_kv_heads ||
        d.head_dim != d0.head_dim || d.ffn != d0.ffn || d.wtype != d0.wtype || d.act != d0.act)
      return fail(QD_ERR_INVALID_ARG, "qd_decode_step: layer %d dims differ from layer 0", i);
  }
  if (!a->embed || !a->final_norm || !a->lm_head || !a->k_cache || !a->v_cache || !a->page_table ||
      !a->rope_table || !a->tok || !a->pos || !a->step || !a->out_tokens || !a->logits || !a->workspace)
    return fail(QD_ERR_INVALID_ARG, "qd_decode_step: null pointer");
  for (int i = 0; i < a->n_layers; ++i)
    if (!a->k_cache[i] || !a->v_cache[i] || !aligned16(a->k_cache[i]) || !aligned16(a->v_cache[i]))
      return fail(QD_ERR_INVALID_ARG, "qd_decode_step: cache %d null or unaligned", i);
  if (a->vocab < 1 || a->max_steps < 1) return fail(QD_ERR_INVALID_ARG, "qd_decode_step: vocab/max_steps");
  if (a->batch < 1 || a->batch > 64)
    return fail(QD_ERR_UNSUPPORTED, "qd_decode_step: batch=%d (supported 1..64)", a->batch);
  if (d0.wtype == QD_W_Q8_0 && a->batch > 1) {
    const int ks[3] = {d0.hidden, d0.n_q_heads * d0.head_dim, d0.ffn};
    for (int k : ks)
      if (!gemm_tc_q8_supported(1, k, a->batch))
        return fail(QD_ERR_UNSUPPORTED, "qd_decode_step: batched Q8_0 K=%d must be a multiple of 256", k);
  }
  if (d0.wtype == QD_W_BF16) {
    const int ks[3] = {d0.hidden, d0.n_q_heads * d0.head_dim, d0.ffn};
    for (int k : ks) {
      if (mma_step(a)) break;
      if (!tc_step(a) && !gemv_bf16_supported(k, a->batch))
        return fail(QD_ERR_UNSUPPORTED, "qd_decode_step: GEMV K=%d with batch %d not supported", k, a->batch);
      if (tc_step(a) && !gemm_tc_supported(1, k, a->batch))
        return fail(QD_ERR_UNSUPPORTED, "qd_decode_step: batched K=%d must be a multiple of 64", k);
    }
  }
  int rc = check_attn_shape("qd_decode_step", a->batch, d0.n_q_heads, d0.n_kv_heads, d0.head_dim, a->page_size,
                            a->max_pages, a->n_pages);
  if (rc) return rc;
  if (a->rope_max_pos < 1) return fail(QD_ERR_INVALID_ARG, "qd_decode_step: rope_max_pos");
  if (d0.wtype == QD_W_INT4 && a->batch != 1)
    return fail(QD_ERR_UNSUPPORTED, "qd_decode_step: INT4 layers run at batch 1");
  if (lm_is_w4(a)) {
    if (a->batch != 1) return fail(QD_ERR_UNSUPPORTED, "qd_decode_step: an INT4 LM head runs at batch 1");
    if (!a->lm_head_scales || ((uintptr_t)a->lm_head_scales & 1u) || !gemv_w4_supported(d0.hidden))
      return fail(QD_ERR_INVALID_ARG, "qd_decode_step: INT4 LM head needs per-row scales and hidden %% 32 == 0");
    if (a->top_k < 0 || a->top_k > 16 || (a->top_k > 0 && (!a->topk_ids || !a->topk_vals)))
      return fail(QD_ERR_INVALID_ARG, "qd_decode_step: top_k=%d (0..16, with topk_ids and topk_vals)", a->top_k);
  }
  const bool q8_head = lm_is_q8(a);
  if (q8_head) {
    if (!gemv_q8_supported(d0.hidden)) return fail(QD_ERR_UNSUPPORTED, "qd_decode_step: Q8_0 head dims");
    if (a->batch > 1 && !tc_step(a))
      return fail(QD_ERR_UNSUPPORTED, "qd_decode_step: a Q8_0 LM head over BF16 layers at batch %d needs the "
                  "tcgen05 step (every K a multiple of 64)", a->batch);
    if (a->batch > 1 && (!gemm_tc_q8_supported(a->vocab, d0.hidden, a->batch) || !aligned16(a->lm_head_scales)))
      return fail(QD_ERR_UNSUPPORTED, "qd_decode_step: batched Q8_0 LM head needs hidden %% 256 == 0");
  }
  if (d0.wtype == QD_W_Q8_0 && a->batch > 1)
    for (int i = 0; i < a->n_layers; ++i) {
      const qd_layer_weights& lw = a->layers[i]->w;
      if (!aligned16(lw.s_qkv) || !aligned16(lw.s_o) || !aligned16(lw.s_gu) || !aligned16(lw.s_down))
        return fail(QD_ERR_INVALID_ARG, "qd_decode_step: batched Q8_0 scales must be 16-byte aligned");
    }
  if (!aligned16(a->embed) || !aligned16(a->lm_head) || !aligned16(a->logits) || !aligned16(a->workspace))
    return fail(QD_ERR_INVALID_ARG, "qd_decode_step: pointers must be 16-byte aligned");
  const StepWs w = step_ws_layout(a, a->workspace);
  if (a->workspace_bytes < w.total)
    return fail(QD_ERR_WORKSPACE, "qd_decode_step: workspace %zu < %zu bytes", a->workspace_bytes, w.total);
  return QD_OK;
}

#define QD_TRY(expr, what)                        \
  do {                                            \
    cudaError_t e_ = (expr);                      \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// Batched decode (BF16: 9..64 sequences; Q8_0: 2..64): every projection is a
// tcgen05 GEMM over the batch (Q8_0 weights widened to bf16 on chip); RMSNorm and
// SwiGLU write the bf16 GEMM operand in small row kernels.
int run_step_tc(const qd_step_args* a, cudaStream_t stream) {
  const qd_layer_dims& d = a->layers[0]->dims;
  const bool q8 = d.wtype == QD_W_Q8_0;
  const StepWs w = step_ws_layout(a, a->workspace);
  const Launch L = make_launch(stream, true);
  const int B = a->batch;
  const int H = d.hidden, F = d.ffn, D = d.head_dim, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int QKV = (Hq + 2 * Hkv) * D;
  // S: the Q8_0 scales of W, or null for bf16 W
  auto gemm = [&](const void* W, const void* S, int R, int K, const void* X, int epi, float* y) {
    GemmTcArgs g = {};
    g.W = W; g.S = S; g.X = X; g.R = R; g.K = K; g.B = B; g.epi = epi; g.y = y;
    g.ws = w.gemm_ws; g.ws_bytes = w.gemm_ws_bytes;
    return launch_gemm_tc(g, L);
  };
  QD_TRY(launch_embed(a->embed, H, a->vocab, a->tok, B, w.res, L), "embed");
  for (int li = 0; li < a->n_layers; ++li) {
    const qd_layer* l = a->layers[li];
    QD_TRY(launch_rmsnorm_rows(w.res, l->w.ln_in, B, H, d.rms_eps, w.xn, L), "rmsnorm");
    QD_TRY(gemm(l->w.w_qkv, q8 ? l->w.s_qkv : nullptr, QKV, H, w.xn, EPI_STORE, w.qkv), "qkv gemm");
    AttnArgs at = {};
    at.qkv = w.qkv; at.q_norm = l->w.q_norm; at.k_norm = l->w.k_norm;
    at.rope = a->rope_table; at.rope_max_pos = a->rope_max_pos; at.eps = d.rms_eps; at.act_bf16 = 1;
    at.pos = a->pos; at.k_pages = a->k_cache[li]; at.v_pages = a->v_cache[li]; at.page_table = a->page_table;
    at.B = B; at.Hq = Hq; at.Hkv = Hkv; at.D = D; at.page_size = a->page_size; at.max_pages = a->max_pages;
    at.n_pages = a->n_pages; at.scale = 1.0f / sqrtf((float)D); at.out_bf16 = w.attn;
    at.workspace = w.attn_ws; at.max_ctx = a->max_pages * a->page_size; at.use_cluster = 0;
    QD_TRY(launch_attention(at, L), "attention");
    QD_TRY(gemm(l->w.w_o, q8 ? l->w.s_o : nullptr, H, Hq * D, w.attn, EPI_RESID_ADD, w.res), "o gemm");
    QD_TRY(launch_rmsnorm_rows(w.res, l->w.ln_post, B, H, d.rms_eps, w.xn, L), "rmsnorm");
    QD_TRY(gemm(l->w.w_gu, q8 ? l->w.s_gu : nullptr, 2 * F, H, w.xn, EPI_STORE, w.gu), "gu gemm");
    QD_TRY(launch_swiglu_rows(w.gu, B, F, w.xn, L), "swiglu");
    QD_TRY(gemm(l->w.w_down, q8 ? l->w.s_down : nullptr, H, F, w.xn, EPI_RESID_ADD, w.res), "down gemm");
  }
  QD_TRY(launch_rmsnorm_rows(w.res, a->final_norm, B, H, d.rms_eps, w.xn, L), "final rmsnorm");
  QD_TRY(gemm(a->lm_head, a->lm_head_scales, a->vocab, H, w.xn, EPI_STORE, a->logits), "lm head gemm");
  QD_TRY(launch_argmax_advance(a->logits, a->vocab, B, a->tok, a->pos, a->step, a->out_tokens, a->max_steps,
                               w.argmax_ws, L),
         "argmax");
  return QD_OK;
}

static int qkv_rows(const qd_layer_dims& d) { return (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim; }

// Small-batch BF16 decode (2..8 sequences): every projection on the mma.sync
// weight-streaming GEMV (the SwiGLU in the gate+up epilogue writing bf16 h), each
// RMSNorm as one row kernel writing bf16 rows (or in the GEMV prologue), paged
// split-KV attention: seven launches per layer (five with the prologue norm).
struct MmaProj {
  const StepTuning& tu;
  int B;
  const Launch& L;
  void* norm_scratch;   // bf16 [B, K] rows for the separate RMSNorm (QD_MMA_NORM_ROWS)
  cudaError_t operator()(const void* W, int R, int K, int pro, const void* x, const void* norm_w, float eps,
                         int epi, float* y, void* y_bf16 = nullptr, L2Prefetch pf = {}) const {
    if (pro == PRO_RMSNORM && mma_norm_rows()) {
      cudaError_t e = launch_rmsnorm_rows((const float*)x, norm_w, B, K, eps, norm_scratch, L);
      if (e != cudaSuccess) return e;
      pro = PRO_X_BF16;
      x = norm_scratch;
    }
    GemvMmaArgs g = {};
    g.W = W; g.R = R; g.K = K; g.B = B; g.pro = pro; g.x = x; g.norm_w = norm_w; g.eps = eps;
    g.epi = epi; g.y = y; g.y_bf16 = y_bf16; g.w_evict_first = tu.w_evict_first;
    g.pf = pf;
    return launch_gemv_mma(g, L);
  }
};

// One layer of the small-batch path over B rows whose residual is w.res. `verify`:
// the B rows are consecutive tokens of one sequence, so all their K/V rows go to the
// cache first and row i attends to positions up to its own. next_w / next_R: the
// GEMV after this layer's down projection (its weights' heads go to L2 early).
int mma_layer(const qd_step_args* a, const qd_layer* l, int li, const StepWs& w, int B, const int32_t* pos,
              const int32_t* page_table, int verify, const MmaProj& proj, const Launch& L, const void* next_w,
              int next_R) {
  const qd_layer_dims& d = l->dims;
  const int H = d.hidden, F = d.ffn, D = d.head_dim, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int QKV = (Hq + 2 * Hkv) * D;
  // head of every CTA span of the next GEMV (R rows of K; the gate+up GEMV's spans are
  // its pair ranges, so the gate half's partition)
  auto tail = [&](const void* Wn, int R, int K) {
    L2Prefetch pf = {};
    if (proj.tu.tail_kb > 0 && Wn) pf = l2_plan_rows(Wn, R, (size_t)K * 2, (size_t)proj.tu.tail_kb << 10);
    return pf;
  };
  QD_TRY(proj(l->w.w_qkv, QKV, H, PRO_RMSNORM, w.res, l->w.ln_in, d.rms_eps, EPI_STORE, w.qkv), "qkv gemv");
  if (verify)
    QD_TRY(launch_kv_write(w.qkv, B, Hq, Hkv, l->w.k_norm, a->rope_table, a->rope_max_pos, d.rms_eps, 1, pos,
                           page_table, a->max_pages, a->page_size, a->max_pages, a->n_pages, a->k_cache[li],
                           a->v_cache[li], L),
           "kv write");
  AttnArgs at = {};
  at.qkv = w.qkv; at.q_norm = l->w.q_norm; at.k_norm = l->w.k_norm;
  at.rope = a->rope_table; at.rope_max_pos = a->rope_max_pos; at.eps = d.rms_eps; at.act_bf16 = 1;
  at.pos = pos; at.k_pages = a->k_cache[li]; at.v_pages = a->v_cache[li]; at.page_table = page_table;
  at.B = B; at.Hq = Hq; at.Hkv = Hkv; at.D = D; at.page_size = a->page_size; at.max_pages = a->max_pages;
  at.n_pages = a->n_pages; at.scale = 1.0f / sqrtf((float)D); at.out_bf16 = w.attn;
  at.workspace = w.attn_ws; at.max_ctx = a->max_pages * a->page_size; at.kv_ready = verify;
  if (verify && verify_attention_supported(B, Hq, Hkv))
    QD_TRY(launch_verify_attention(at, B, L), "verify attention");
  else
    QD_TRY(launch_attention(at, L), "attention");
  QD_TRY(proj(l->w.w_o, H, Hq * D, PRO_X_BF16, w.attn, nullptr, 0.f, EPI_RESID_ADD, w.res, nullptr,
              tail(l->w.w_gu, F, H)),
         "o gemv");
  QD_TRY(proj(l->w.w_gu, 2 * F, H, PRO_RMSNORM, w.res, l->w.ln_post, d.rms_eps, EPI_SWIGLU, nullptr, w.xn,
              tail(l->w.w_down, H, F)),
         "gu gemv");
  QD_TRY(proj(l->w.w_down, H, F, PRO_X_BF16, w.xn, nullptr, 0.f, EPI_RESID_ADD, w.res, nullptr,
              tail(next_w, next_R, H)),
         "down gemv");
  return QD_OK;
}

int run_step_mma(const qd_step_args* a, cudaStream_t stream) {
  const qd_layer_dims& d = a->layers[0]->dims;
  const StepWs w = step_ws_layout(a, a->workspace);
  const Launch L = make_launch(stream, true);
  const int B = a->batch;
  const MmaProj proj{step_tuning(), B, L, w.gu};
  QD_TRY(launch_embed(a->embed, d.hidden, a->vocab, a->tok, B, w.res, L), "embed");
  for (int li = 0; li < a->n_layers; ++li) {
    const bool last = li + 1 == a->n_layers;
    const int rc = mma_layer(a, a->layers[li], li, w, B, a->pos, a->page_table, 0, proj, L,
                             last ? a->lm_head : a->layers[li + 1]->w.w_qkv, last ? a->vocab : qkv_rows(d));
    if (rc) return rc;
  }
  QD_TRY(proj(a->lm_head, a->vocab, d.hidden, PRO_RMSNORM, w.res, a->final_norm, d.rms_eps, EPI_STORE, a->logits),
         "lm head gemv");
  QD_TRY(launch_argmax_advance(a->logits, a->vocab, B, a->tok, a->pos, a->step, a->out_tokens, a->max_steps,
                               w.argmax_ws, L),
         "argmax");
  return QD_OK;
}

// The INT4 LM head of a batch-1 step: the GEMV, its top-k and the argmax advance in
// one launch.
cudaError_t launch_lm_head_w4(const qd_step_args* a, const StepWs& w, const Launch& L) {
  GemvW4Args g = {};
  g.W = a->lm_head; g.d = a->lm_head_scales; g.R = a->vocab; g.K = a->layers[0]->dims.hidden;
  g.pro = PRO_RMSNORM; g.x = w.res; g.norm_w = a->final_norm; g.eps = a->layers[0]->dims.rms_eps;
  g.epi = EPI_TOPK; g.y = a->logits; g.w_evict_first = step_tuning().w_evict_first;
  g.top_k = a->top_k > 0 ? a->top_k : 1; g.ws = w.topk_ws;
  g.tok = a->tok; g.pos = a->pos; g.step = a->step; g.out_tokens = a->out_tokens; g.max_steps = a->max_steps;
  g.topk_ids = a->top_k > 0 ? a->topk_ids : nullptr; g.topk_vals = a->top_k > 0 ? a->topk_vals : nullptr;
  return launch_gemv_w4(g, L);
}

// Batch-1 step of INT4 (W4A16) layers: the BF16 step's order with the W4A16 GEMVs
// (bf16 activations: the same rounding points as the BF16 model).
int run_step_w4(const qd_step_args* a, cudaStream_t stream) {
  const qd_layer_dims& d = a->layers[0]->dims;
  const StepWs w = step_ws_layout(a, a->workspace);
  const Launch L = make_launch(stream, true);
  const int H = d.hidden, F = d.ffn, D = d.head_dim, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int QKV = (Hq + 2 * Hkv) * D;
  const int wef = step_tuning().w_evict_first;
  auto gemv = [&](const void* W, const void* S, int R, int K, int pro, const void* x, const void* nw, int epi,
                  float* y, void* y_bf16) {
    GemvW4Args g = {};
    g.W = W; g.d = S; g.R = R; g.K = K; g.pro = pro; g.x = x; g.norm_w = nw; g.eps = d.rms_eps; g.epi = epi;
    g.y = y; g.y_bf16 = y_bf16; g.w_evict_first = wef;
    g.split_ws = w.w4_ws; g.split_ws_bytes = w.w4_ws_bytes;
    return launch_gemv_w4(g, L);
  };
  QD_TRY(launch_embed(a->embed, H, a->vocab, a->tok, 1, w.res, L), "embed");
  for (int li = 0; li < a->n_layers; ++li) {
    const qd_layer* l = a->layers[li];
    QD_TRY(gemv(l->w.w_qkv, l->w.s_qkv, QKV, H, PRO_RMSNORM, w.res, l->w.ln_in, EPI_STORE, w.qkv, nullptr),
           "qkv gemv w4");
    AttnArgs at = {};
    at.qkv = w.qkv; at.q_norm = l->w.q_norm; at.k_norm = l->w.k_norm;
    at.rope = a->rope_table; at.rope_max_pos = a->rope_max_pos; at.eps = d.rms_eps; at.act_bf16 = 1;
    at.pos = a->pos; at.k_pages = a->k_cache[li]; at.v_pages = a->v_cache[li]; at.page_table = a->page_table;
    at.B = 1; at.Hq = Hq; at.Hkv = Hkv; at.D = D; at.page_size = a->page_size; at.max_pages = a->max_pages;
    at.n_pages = a->n_pages; at.scale = 1.0f / sqrtf((float)D); at.out_bf16 = w.attn;
    at.workspace = w.attn_ws; at.max_ctx = a->max_pages * a->page_size;
    QD_TRY(launch_attention(at, L), "attention");
    QD_TRY(gemv(l->w.w_o, l->w.s_o, H, Hq * D, PRO_X_BF16, w.attn, nullptr, EPI_RESID_ADD, w.res, nullptr),
           "o gemv w4");
    QD_TRY(gemv(l->w.w_gu, l->w.s_gu, 2 * F, H, PRO_RMSNORM, w.res, l->w.ln_post, EPI_SWIGLU, nullptr, w.xn),
           "gu gemv w4");
    QD_TRY(gemv(l->w.w_down, l->w.s_down, H, F, PRO_X_BF16, w.xn, nullptr, EPI_RESID_ADD, w.res, nullptr),
           "down gemv w4");
  }
  if (lm_is_w4(a)) {
    QD_TRY(launch_lm_head_w4(a, w, L), "lm head w4");
    return QD_OK;
  }
  if (lm_is_q8(a)) {
    GemvQ8Args g = {};
    g.qs = (const int8_t*)a->lm_head; g.d = a->lm_head_scales; g.R = a->vocab; g.K = H; g.act = a->lm_act;
    g.pro = PRO_RMSNORM; g.x = w.res; g.norm_w = a->final_norm; g.eps = d.rms_eps; g.epi = EPI_STORE; g.y = a->logits;
    g.claim = w.claims + 2 * 5 * a->n_layers;
    QD_TRY(launch_gemv_q8(g, L), "lm head q8");
  } else {
    GemvBf16Args g = {};
    g.W = a->lm_head; g.R = a->vocab; g.K = H; g.batch = 1; g.pro = PRO_RMSNORM; g.x = w.res;
    g.norm_w = a->final_norm; g.eps = d.rms_eps; g.epi = EPI_STORE; g.y = a->logits;
    QD_TRY(launch_gemv_bf16(g, L), "lm head");
  }
  QD_TRY(launch_argmax_advance(a->logits, a->vocab, 1, a->tok, a->pos, a->step, a->out_tokens, a->max_steps,
                               w.argmax_ws, L),
         "argmax");
  return QD_OK;
}

int run_step(const qd_step_args* a, cudaStream_t stream) {
  if (mma_step(a)) return run_step_mma(a, stream);
  if (tc_step(a)) return run_step_tc(a, stream);
  if (a->layers[0]->dims.wtype == QD_W_INT4) return run_step_w4(a, stream);
  const qd_layer_dims& d = a->layers[0]->dims;
  const StepWs w = step_ws_layout(a, a->workspace);
  if (!step_kernels_forced()) {
    std::vector<StreamLayerPtrs> lp;
    StreamStepArgs sa;
    if (stream_args(a, w, lp, sa)) {
      QD_TRY(launch_stream_step(sa, make_launch(stream, false)), "persistent step");
      return QD_OK;
    }
  }
  const Launch L = make_launch(stream, true);
  const int B = a->batch;
  const int H = d.hidden, F = d.ffn, D = d.head_dim, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int QKV = (Hq + 2 * Hkv) * D;
  const bool q8 = d.wtype == QD_W_Q8_0;
  const StepTuning& pft = step_tuning();
  // batch 1 on the ring GEMV: SwiGLU in the gate+up epilogue (bf16 h), so the down
  // projection reads 2F bytes of h instead of 8F of gate/up and recomputes nothing
  const bool swiglu_epi = !q8 && B == 1 && gemv_bf16_swiglu_ok(H) && gemv_bf16_ring_ok(F, 1) &&
                          !pft.swiglu_in_down;
  const bool q8_swiglu_epi = q8 && B == 1 && gemv_q8_swiglu_ok(H) && gemv_q8_supported(F) && !pft.swiglu_in_down;
  // each batch-1 Q8_0 GEMV launch of the step owns a pair of row-claim counters
  auto claim = [&](int li, int k) { return B == 1 ? w.claims + 2 * (5 * li + k) : nullptr; };
  // head of every span of the next batch-1 BF16 GEMV (R rows of K), or nothing
  auto tail_plan = [&](const void* Wn, int R, int K) {
    L2Prefetch pf = {};
    if (B == 1 && pft.tail_kb > 0) pf = l2_plan_rows(Wn, R, (size_t)K * 2, (size_t)pft.tail_kb << 10);
    return pf;
  };

  QD_TRY(launch_embed(a->embed, H, a->vocab, a->tok, B, w.res, L), "embed");
  for (int li = 0; li < a->n_layers; ++li) {
    const qd_layer* l = a->layers[li];
    // QKV projection, RMSNorm(res; ln_in) fused into the prologue
    if (q8) {
      GemvQ8Args g = {};
      g.w_evict_first = pft.w_evict_first;
      g.claim = claim(li, 0);
      g.qs = (const int8_t*)l->w.w_qkv; g.d = l->w.s_qkv; g.R = QKV; g.K = H; g.act = d.act;
      g.pro = PRO_RMSNORM; g.x = w.res; g.norm_w = l->w.ln_in; g.eps = d.rms_eps; g.epi = EPI_STORE; g.y = w.qkv;
      QD_TRY(launch_gemv_q8(g, L), "qkv gemv q8");
    } else {
      GemvBf16Args g = {};
      g.w_evict_first = pft.w_evict_first;
      g.ring_kb = pft.qkv_ring_kb;
      g.W = l->w.w_qkv; g.R = QKV; g.K = H; g.batch = B; g.pro = PRO_RMSNORM; g.x = w.res;
      g.norm_w = l->w.ln_in; g.eps = d.rms_eps; g.epi = EPI_STORE; g.y = w.qkv;
      QD_TRY(launch_gemv_bf16(g, L), "qkv gemv");
    }
    // QK-norm + RoPE + K/V cache write + split-KV attention + combine
    AttnArgs at = {};
    at.qkv = w.qkv; at.q_norm = l->w.q_norm; at.k_norm = l->w.k_norm;
    at.rope = a->rope_table; at.rope_max_pos = a->rope_max_pos; at.eps = d.rms_eps; at.act_bf16 = !q8;
    at.pos = a->pos; at.k_pages = a->k_cache[li]; at.v_pages = a->v_cache[li]; at.page_table = a->page_table;
    at.B = B; at.Hq = Hq; at.Hkv = Hkv; at.D = D; at.page_size = a->page_size; at.max_pages = a->max_pages;
    at.n_pages = a->n_pages; at.scale = 1.0f / sqrtf((float)D);
    if (q8) at.out_f32 = (float*)w.attn;
    else at.out_bf16 = w.attn;
    at.workspace = w.attn_ws; at.max_ctx = a->max_pages * a->page_size; at.use_cluster = attn_cluster_enabled();
    if (!q8 && B == 1) {
      if (pft.attn_wo_kb) at.pf[0] = l2_plan_rows(l->w.w_o, H, (size_t)Hq * D * 2, (size_t)pft.attn_wo_kb << 10);
      at.pf_late = pft.attn_late;
      at.trig_loop = pft.attn_trig_loop;
      if (pft.kv_pf) {  // the last layer fetches layer 0's rows for the next step
        const int ln = li + 1 < a->n_layers ? li + 1 : 0;
        at.k_next = a->k_cache[ln];
        at.v_next = a->v_cache[ln];
        at.kv_pf = pft.kv_pf;
      }
      if (pft.attn_gu_kb) at.pf[1] = l2_plan_rows(l->w.w_gu, 2 * F, (size_t)H * 2, (size_t)pft.attn_gu_kb << 10);
    }
    QD_TRY(launch_attention(at, L), "attention");
    // O projection + residual add
    if (q8) {
      GemvQ8Args g = {};
      g.w_evict_first = pft.w_evict_first;
      g.claim = claim(li, 1);
      g.qs = (const int8_t*)l->w.w_o; g.d = l->w.s_o; g.R = H; g.K = Hq * D; g.act = d.act;
      g.pro = PRO_X_F32; g.x = w.attn; g.epi = EPI_RESID_ADD; g.y = w.res;
      QD_TRY(launch_gemv_q8(g, L), "o gemv q8");
    } else {
      GemvBf16Args g = {};
      g.w_evict_first = pft.w_evict_first;
      g.W = l->w.w_o; g.R = H; g.K = Hq * D; g.batch = B; g.pro = PRO_X_BF16; g.x = w.attn;
      g.epi = EPI_RESID_ADD; g.y = w.res;
      g.pf = tail_plan(l->w.w_gu, 2 * F, H);
      g.ring_kb = pft.o_ring_kb;
      QD_TRY(launch_gemv_bf16(g, L), "o gemv");
    }
    // gate+up projection, RMSNorm(res; ln_post) fused into the prologue
    if (q8) {
      GemvQ8Args g = {};
      g.w_evict_first = pft.w_evict_first;
      g.claim = claim(li, 2);
      g.qs = (const int8_t*)l->w.w_gu; g.d = l->w.s_gu; g.R = 2 * F; g.K = H; g.act = d.act;
      g.pro = PRO_RMSNORM; g.x = w.res; g.norm_w = l->w.ln_post; g.eps = d.rms_eps; g.epi = EPI_STORE; g.y = w.gu;
      if (q8_swiglu_epi) g.epi = EPI_SWIGLU;  // y = f32 silu(gate) * up [F]
      QD_TRY(launch_gemv_q8(g, L), "gu gemv q8");
    } else {
      GemvBf16Args g = {};
      g.w_evict_first = pft.w_evict_first;
      g.W = l->w.w_gu; g.R = 2 * F; g.K = H; g.batch = B; g.pro = PRO_RMSNORM; g.x = w.res;
      g.norm_w = l->w.ln_post; g.eps = d.rms_eps; g.epi = EPI_STORE; g.y = w.gu;
      if (swiglu_epi) {  // h = bf16(silu(gate) * up) formed in the epilogue, into xn
        g.epi = EPI_SWIGLU; g.y = nullptr; g.y_bf16 = w.xn;
      }
      g.pf = tail_plan(l->w.w_down, H, F);
      QD_TRY(launch_gemv_bf16(g, L), "gu gemv");
    }
    // down projection with SwiGLU formed on load, + residual add
    if (q8) {
      GemvQ8Args g = {};
      g.w_evict_first = pft.w_evict_first;
      g.claim = claim(li, 3);
      g.qs = (const int8_t*)l->w.w_down; g.d = l->w.s_down; g.R = H; g.K = F; g.act = d.act;
      g.pro = PRO_SWIGLU; g.x = w.gu; g.epi = EPI_RESID_ADD; g.y = w.res;
      if (q8_swiglu_epi) g.pro = PRO_X_F32;  // the gate+up epilogue already formed silu(g) * u
      QD_TRY(launch_gemv_q8(g, L), "down gemv q8");
    } else {
      GemvBf16Args g = {};
      g.w_evict_first = pft.w_evict_first;
      g.ring_kb = pft.down_ring_kb;
      g.W = l->w.w_down; g.R = H; g.K = F; g.batch = B; g.pro = PRO_SWIGLU; g.x = w.gu;
      g.epi = EPI_RESID_ADD; g.y = w.res;
      if (swiglu_epi) { g.pro = PRO_X_BF16; g.x = w.xn; }
      if (li + 1 < a->n_layers) g.pf = tail_plan(a->layers[li + 1]->w.w_qkv, QKV, H);
      else if (!a->lm_head_scales) g.pf = tail_plan(a->lm_head, a->vocab, H);
      if (li + 1 == a->n_layers && lm_is_w4(a)) g.pf = L2Prefetch{};
      QD_TRY(launch_gemv_bf16(g, L), "down gemv");
    }
  }
  // final RMSNorm + LM head
  if (lm_is_w4(a)) {
    QD_TRY(launch_lm_head_w4(a, w, L), "lm head w4");
    return QD_OK;
  }
  if (a->lm_head_scales) {
    GemvQ8Args g = {};
    g.w_evict_first = pft.w_evict_first;
    g.claim = claim(a->n_layers, 0);
    g.qs = (const int8_t*)a->lm_head; g.d = a->lm_head_scales; g.R = a->vocab; g.K = H; g.act = a->lm_act;
    g.pro = PRO_RMSNORM; g.x = w.res; g.norm_w = a->final_norm; g.eps = d.rms_eps; g.epi = EPI_STORE; g.y = a->logits;
    QD_TRY(launch_gemv_q8(g, L), "lm head q8");
  } else {
    GemvBf16Args g = {};
    g.w_evict_first = pft.w_evict_first;
    g.W = a->lm_head; g.R = a->vocab; g.K = H; g.batch = B; g.pro = PRO_RMSNORM; g.x = w.res;
    g.norm_w = a->final_norm; g.eps = d.rms_eps; g.epi = EPI_STORE; g.y = a->logits;
    QD_TRY(launch_gemv_bf16(g, L), "lm head");
  }
  QD_TRY(launch_argmax_advance(a->logits, a->vocab, B, a->tok, a->pos, a->step, a->out_tokens, a->max_steps,
                               w.argmax_ws, L),
         "argmax");
  return QD_OK;
}

// ------------------------------------------------------------------ speculative verify
// k rows of one sequence: the batched step's buffers for k rows (its projections on the
// tcgen05 GEMMs), then the rows' tokens, positions, page-table rows and argmax scratch.
struct VerifyWs {
  StepWs w;
  int32_t* tokens;   // [k]
  int32_t* vpos;     // [k]
  int32_t* vpt;      // [k, max_pages]
  int32_t* scratch;  // [3k]: argmax position, step, output slot
  size_t total;
};

// The verify and prefill scratch follows the decode step's own workspace, so the
// step's counters (zero between launches) are never overwritten by a pass.
VerifyWs verify_ws_layout(const qd_step_args* a, int k, void* base) {
  qd_step_args ak = *a;
  ak.batch = k;
  VerifyWs v;
  const size_t step_bytes = step_ws_layout(a, nullptr).total;
  unsigned char* p = (unsigned char*)base + step_bytes;
  v.w = step_ws_layout_for(&ak, p, true);
  size_t off = v.w.total;
  v.tokens = (int32_t*)(p + off); off += al256((size_t)k * 4);
  v.vpos = (int32_t*)(p + off); off += al256((size_t)k * 4);
  v.vpt = (int32_t*)(p + off); off += al256((size_t)k * a->max_pages * 4);
  v.scratch = (int32_t*)(p + off); off += al256((size_t)3 * k * 4);
  v.total = step_bytes + off;
  return v;
}

constexpr int kMaxVerify = 8;

// A verify pass on the mma.sync GEMVs: the small-batch step's rule for k rows (k = 1
// included: the GEMV takes one row as well).
bool mma_verify(const qd_step_args* a, int k) {
  qd_step_args ak = *a;
  ak.batch = std::max(k, 2);
  return mma_step(&ak);
}

int validate_verify(const qd_step_args* a, const int32_t* draft, int k, const float* logits, const int32_t* target,
                    const int32_t* n_accept) {
  if (!a) return fail(QD_ERR_INVALID_ARG, "qd_verify_step: null args");
  if (a->batch != 1) return fail(QD_ERR_UNSUPPORTED, "qd_verify_step: one sequence (batch 1)");
  if (k < 1 || k > kMaxVerify) return fail(QD_ERR_INVALID_ARG, "qd_verify_step: k=%d (1..%d)", k, kMaxVerify);
  if ((k > 1 && !draft) || !logits || !target || !n_accept)
    return fail(QD_ERR_INVALID_ARG, "qd_verify_step: null pointer");
  if (!aligned16(logits)) return fail(QD_ERR_INVALID_ARG, "qd_verify_step: logits must be 16-byte aligned");
  int rc = validate_step(a);
  if (rc) return rc;
  const qd_layer_dims& d = a->layers[0]->dims;
  if (d.wtype == QD_W_INT4 || lm_is_w4(a))
    return fail(QD_ERR_UNSUPPORTED, "qd_verify_step: INT4 weights run the batch-1 GEMV path only");
  const bool q8 = d.wtype == QD_W_Q8_0;
  const int ks[3] = {d.hidden, d.n_q_heads * d.head_dim, d.ffn};
  for (int K : ks)
    if (!mma_verify(a, k) && (q8 ? !gemm_tc_q8_supported(1, K, k) : !gemm_tc_supported(1, K, k)))
      return fail(QD_ERR_UNSUPPORTED, "qd_verify_step: projection K=%d needs a multiple of %d", K, q8 ? 256 : 64);
  if (a->lm_head_scales && !gemm_tc_q8_supported(a->vocab, d.hidden, k))
    return fail(QD_ERR_UNSUPPORTED, "qd_verify_step: Q8_0 LM head needs hidden %% 256 == 0");
  if (q8)
    for (int i = 0; i < a->n_layers; ++i) {
      const qd_layer_weights& lw = a->layers[i]->w;
      if (!aligned16(lw.s_qkv) || !aligned16(lw.s_o) || !aligned16(lw.s_gu) || !aligned16(lw.s_down))
        return fail(QD_ERR_INVALID_ARG, "qd_verify_step: Q8_0 scales must be 16-byte aligned");
    }
  const VerifyWs v = verify_ws_layout(a, k, a->workspace);
  if (a->workspace_bytes < v.total)
    return fail(QD_ERR_WORKSPACE, "qd_verify_step: workspace %zu < %zu bytes", a->workspace_bytes, v.total);
  return QD_OK;
}

int run_verify(const qd_step_args* a, const int32_t* draft, int k, float* logits, int32_t* target,
               int32_t* n_accept, cudaStream_t stream) {
  const qd_layer_dims& d = a->layers[0]->dims;
  const bool q8 = d.wtype == QD_W_Q8_0;
  const VerifyWs v = verify_ws_layout(a, k, a->workspace);
  const StepWs& w = v.w;
  const Launch L = make_launch(stream, true);
  const int H = d.hidden, F = d.ffn, D = d.head_dim, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int QKV = (Hq + 2 * Hkv) * D;
  auto gemm = [&](const void* W, const void* S, int R, int K, const void* X, int epi, float* y) {
    GemmTcArgs g = {};
    g.W = W; g.S = S; g.X = X; g.R = R; g.K = K; g.B = k; g.epi = epi; g.y = y;
    g.ws = w.gemm_ws; g.ws_bytes = w.gemm_ws_bytes;
    return launch_gemm_tc(g, L);
  };
  QD_TRY(launch_verify_prep(a->tok, a->pos, draft, k, a->page_table, a->max_pages, v.tokens, v.vpos, v.vpt,
                            v.scratch, L),
         "verify prep");
  QD_TRY(launch_embed(a->embed, H, a->vocab, v.tokens, k, w.res, L), "embed");
  const bool mma = mma_verify(a, k);
  const MmaProj proj{step_tuning(), k, L, w.gu};
  for (int li = 0; li < a->n_layers && mma; ++li) {
    const bool last = li + 1 == a->n_layers;
    const int rc = mma_layer(a, a->layers[li], li, w, k, v.vpos, v.vpt, 1, proj, L,
                             last ? a->lm_head : a->layers[li + 1]->w.w_qkv, last ? a->vocab : qkv_rows(d));
    if (rc) return rc;
  }
  if (mma)
    QD_TRY(proj(a->lm_head, a->vocab, H, PRO_RMSNORM, w.res, a->final_norm, d.rms_eps, EPI_STORE, logits),
           "lm head gemv");
  for (int li = 0; li < a->n_layers && !mma; ++li) {
    const qd_layer* l = a->layers[li];
    QD_TRY(launch_rmsnorm_rows(w.res, l->w.ln_in, k, H, d.rms_eps, w.xn, L), "rmsnorm");
    QD_TRY(gemm(l->w.w_qkv, q8 ? l->w.s_qkv : nullptr, QKV, H, w.xn, EPI_STORE, w.qkv), "qkv gemm");
    // all k rows' K/V go to the cache first, so row i attends to rows pos .. pos + i
    QD_TRY(launch_kv_write(w.qkv, k, Hq, Hkv, l->w.k_norm, a->rope_table, a->rope_max_pos, d.rms_eps, 1, v.vpos,
                           v.vpt, a->max_pages, a->page_size, a->max_pages, a->n_pages, a->k_cache[li],
                           a->v_cache[li], L),
           "kv write");
    AttnArgs at = {};
    at.qkv = w.qkv; at.q_norm = l->w.q_norm; at.k_norm = l->w.k_norm;
    at.rope = a->rope_table; at.rope_max_pos = a->rope_max_pos; at.eps = d.rms_eps; at.act_bf16 = 1;
    at.pos = v.vpos; at.k_pages = a->k_cache[li]; at.v_pages = a->v_cache[li]; at.page_table = v.vpt;
    at.B = k; at.Hq = Hq; at.Hkv = Hkv; at.D = D; at.page_size = a->page_size; at.max_pages = a->max_pages;
    at.n_pages = a->n_pages; at.scale = 1.0f / sqrtf((float)D); at.out_bf16 = w.attn;
    at.workspace = w.attn_ws; at.max_ctx = a->max_pages * a->page_size; at.kv_ready = 1;
    if (verify_attention_supported(k, Hq, Hkv))
      QD_TRY(launch_verify_attention(at, k, L), "verify attention");
    else
      QD_TRY(launch_attention(at, L), "attention");
    QD_TRY(gemm(l->w.w_o, q8 ? l->w.s_o : nullptr, H, Hq * D, w.attn, EPI_RESID_ADD, w.res), "o gemm");
    QD_TRY(launch_rmsnorm_rows(w.res, l->w.ln_post, k, H, d.rms_eps, w.xn, L), "rmsnorm");
    QD_TRY(gemm(l->w.w_gu, q8 ? l->w.s_gu : nullptr, 2 * F, H, w.xn, EPI_STORE, w.gu), "gu gemm");
    QD_TRY(launch_swiglu_rows(w.gu, k, F, w.xn, L), "swiglu");
    QD_TRY(gemm(l->w.w_down, q8 ? l->w.s_down : nullptr, H, F, w.xn, EPI_RESID_ADD, w.res), "down gemm");
  }
  if (!mma) {
    QD_TRY(launch_rmsnorm_rows(w.res, a->final_norm, k, H, d.rms_eps, w.xn, L), "final rmsnorm");
    QD_TRY(gemm(a->lm_head, a->lm_head_scales, a->vocab, H, w.xn, EPI_STORE, logits), "lm head gemm");
  }
  QD_TRY(launch_argmax_advance(logits, a->vocab, k, target, v.scratch, v.scratch + k, v.scratch + 2 * k, 1,
                               w.argmax_ws, L),
         "argmax");
  QD_TRY(launch_verify_accept(draft, target, k, a->tok, a->pos, a->step, a->out_tokens, a->max_steps, n_accept, L),
         "accept");
  return QD_OK;
}

// ---- prefill: the prompt's n tokens of one sequence through every layer at once
struct PrefillWs {
  float* res;        // [n, H]
  float* qkv;        // [n, QKV]
  void* attn;        // bf16 [n, Hq D]
  float* gu;         // [n, 2F]
  void* xn;          // bf16 [n, max(H, F)]
  int32_t* vpos;     // [n] positions of the rows
  void* argmax_ws;
  void* kv_pack;     // the tcgen05 attention's packed K / V copies
  size_t kv_pack_bytes;
  void* wide_w;      // Q8_0 above prefill_widen_rows() rows: bf16 copy of one projection's weights
  size_t total;
};

// Q8_0 prefill of more rows than this: each projection's weights are widened to bf16
// once (bf16(f32(d) q), the tensor-core lane's own widening) and the rows run on the
// bf16 GEMMs, which are compute-bound there; up to it the Q8_0 GEMM, which reads 1.0625
// bytes per weight, is the faster one. QD_PREFILL_WIDEN_ROWS overrides it, read once per
// process so that the workspace size and the pass agree.
int prefill_widen_rows() {
  static const int v = [] {
    const char* e = getenv("QD_PREFILL_WIDEN_ROWS");
    return e ? std::max(0, atoi(e)) : 128;
  }();
  return v;
}

constexpr int kMaxPrefill = 32768;

PrefillWs prefill_ws_layout(const qd_step_args* a, int n, void* base) {
  const qd_layer_dims& d = a->layers[0]->dims;
  const size_t qkv = (size_t)(d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim;
  const size_t step_bytes = step_ws_layout(a, nullptr).total;
  unsigned char* p = (unsigned char*)base + step_bytes;
  PrefillWs w;
  size_t off = 0;
  w.res = (float*)(p + off); off += al256((size_t)n * d.hidden * 4);
  w.qkv = (float*)(p + off); off += al256((size_t)n * qkv * 4);
  w.attn = (void*)(p + off); off += al256((size_t)n * d.n_q_heads * d.head_dim * 2);
  w.gu = (float*)(p + off); off += al256((size_t)n * 2 * d.ffn * 4);
  w.xn = (void*)(p + off); off += al256((size_t)n * std::max(d.hidden, d.ffn) * 2);
  w.vpos = (int32_t*)(p + off); off += al256((size_t)n * 4);
  w.argmax_ws = (void*)(p + off); off += al256(argmax_workspace_bytes(1));
  w.kv_pack = (void*)(p + off);
  w.kv_pack_bytes = prefill_attention_tc_scratch_bytes(d.n_kv_heads, a->max_pages * a->page_size);
  off += al256(w.kv_pack_bytes);
  w.wide_w = nullptr;
  if (d.wtype == QD_W_Q8_0 && n > prefill_widen_rows()) {
    const size_t H = d.hidden, F = d.ffn, A = (size_t)d.n_q_heads * d.head_dim;
    const size_t most = std::max(std::max(qkv * H, H * A), std::max(2 * F * H, H * F));
    w.wide_w = (void*)(p + off);
    off += al256(most * 2);
  }
  w.total = step_bytes + off;
  return w;
}

int validate_prefill(const qd_step_args* a, const int32_t* tokens, int n, const float* logits) {
  if (!a) return fail(QD_ERR_INVALID_ARG, "qd_prefill: null args");
  if (a->batch != 1) return fail(QD_ERR_UNSUPPORTED, "qd_prefill: one sequence (batch 1)");
  if (n < 1 || n > kMaxPrefill) return fail(QD_ERR_INVALID_ARG, "qd_prefill: n_tokens=%d (1..%d)", n, kMaxPrefill);
  if (!tokens || !logits) return fail(QD_ERR_INVALID_ARG, "qd_prefill: null pointer");
  if (!aligned16(logits)) return fail(QD_ERR_INVALID_ARG, "qd_prefill: logits must be 16-byte aligned");
  int rc = validate_step(a);
  if (rc) return rc;
  const qd_layer_dims& d = a->layers[0]->dims;
  if (d.wtype == QD_W_INT4 || lm_is_w4(a))
    return fail(QD_ERR_UNSUPPORTED, "qd_prefill: INT4 weights run the batch-1 GEMV path only");
  const bool q8 = d.wtype == QD_W_Q8_0;
  const int ks[3] = {d.hidden, d.n_q_heads * d.head_dim, d.ffn};
  for (int K : ks)
    if (!gemm_tc_rows_supported(1, K, n, q8) || (n <= 64 && !(q8 ? gemm_tc_q8_supported(1, K, n)
                                                                 : gemm_tc_supported(1, K, n))))
      return fail(QD_ERR_UNSUPPORTED, "qd_prefill: projection K=%d needs a multiple of %d", K, q8 ? 256 : 64);
  if (a->lm_head_scales && !gemm_tc_q8_supported(a->vocab, d.hidden, 1))
    return fail(QD_ERR_UNSUPPORTED, "qd_prefill: Q8_0 LM head needs hidden %% 256 == 0");
  if (q8)
    for (int i = 0; i < a->n_layers; ++i) {
      const qd_layer_weights& lw = a->layers[i]->w;
      if (!aligned16(lw.s_qkv) || !aligned16(lw.s_o) || !aligned16(lw.s_gu) || !aligned16(lw.s_down))
        return fail(QD_ERR_INVALID_ARG, "qd_prefill: Q8_0 scales must be 16-byte aligned");
    }
  const PrefillWs w = prefill_ws_layout(a, n, a->workspace);
  if (a->workspace_bytes < w.total)
    return fail(QD_ERR_WORKSPACE, "qd_prefill: workspace %zu < %zu bytes", a->workspace_bytes, w.total);
  return QD_OK;
}

int run_prefill(const qd_step_args* a, const int32_t* tokens, int n, float* logits, cudaStream_t stream) {
  const qd_layer_dims& d = a->layers[0]->dims;
  const bool q8 = d.wtype == QD_W_Q8_0;
  const PrefillWs w = prefill_ws_layout(a, n, a->workspace);
  const Launch L = make_launch(stream, true);
  const int H = d.hidden, F = d.ffn, D = d.head_dim, Hq = d.n_q_heads, Hkv = d.n_kv_heads;
  const int QKV = (Hq + 2 * Hkv) * D;
  auto gemm = [&](const void* W, const void* S, int R, int K, const void* X, int B, int epi, float* y) {
    GemmTcArgs g = {};
    g.W = W; g.S = S; g.X = X; g.R = R; g.K = K; g.B = B; g.epi = epi; g.y = y;
    return launch_gemm_tc(g, L);
  };
  // Q8_0 over many rows: widen the projection's weights into w.wide_w, then the bf16
  // GEMM. The GEMM issues its first weight loads before its dependency wait, so it
  // launches without the programmatic dependency (it starts once the widening is done);
  // the widening itself waits for the kernels before it, the last reader of w.wide_w
  // among them, before its first store.
  const bool widen = w.wide_w != nullptr;
  const Launch L_full = make_launch(stream, false);
  auto widened = [&](const void* W, const void* S, int R, int K) -> cudaError_t {
    return launch_q8_widen(W, S, R, K, w.wide_w, L);
  };
  auto proj = [&](const void* W, const void* S, int R, int K, const void* X, int epi, float* y) -> cudaError_t {
    if (!widen) return gemm(W, S, R, K, X, n, epi, y);
    cudaError_t e = widened(W, S, R, K);
    if (e != cudaSuccess) return e;
    GemmTcArgs g = {};
    g.W = w.wide_w; g.X = X; g.R = R; g.K = K; g.B = n; g.epi = epi; g.y = y;
    return launch_gemm_tc(g, L_full);
  };
  // QD_PREFILL_ATTN (read per call): "mma" keeps the attention on the mma.sync kernel;
  // otherwise tcgen05 (2048 / 4096-token prefill 53.0K / 44.0K -> 60.4K / 54.7K tok/s)
  const char* pa = getenv("QD_PREFILL_ATTN");
  const bool tc_attn = !(pa && strcmp(pa, "mma") == 0);
  QD_TRY(launch_prefill_prep(a->pos, n, w.vpos, L), "prefill prep");
  QD_TRY(launch_embed(a->embed, H, a->vocab, tokens, n, w.res, L), "embed");
  for (int li = 0; li < a->n_layers; ++li) {
    const qd_layer* l = a->layers[li];
    QD_TRY(launch_rmsnorm_rows(w.res, l->w.ln_in, n, H, d.rms_eps, w.xn, L), "rmsnorm");
    QD_TRY(proj(l->w.w_qkv, q8 ? l->w.s_qkv : nullptr, QKV, H, w.xn, EPI_STORE, w.qkv), "qkv gemm");
    // every row's K/V reaches the cache before the attention reads keys up to its own position
    QD_TRY(launch_kv_write(w.qkv, n, Hq, Hkv, l->w.k_norm, a->rope_table, a->rope_max_pos, d.rms_eps, 1, w.vpos,
                           a->page_table, 0, a->page_size, a->max_pages, a->n_pages, a->k_cache[li],
                           a->v_cache[li], L),
           "kv write");
    PrefillAttnArgs at = {};
    at.qkv = w.qkv; at.n = n; at.Hq = Hq; at.Hkv = Hkv; at.D = D; at.q_norm = l->w.q_norm;
    at.rope = a->rope_table; at.rope_max_pos = a->rope_max_pos; at.eps = d.rms_eps; at.act_bf16 = 1;
    at.pos = a->pos; at.k_pages = a->k_cache[li]; at.v_pages = a->v_cache[li]; at.page_table = a->page_table;
    at.page_size = a->page_size; at.max_pages = a->max_pages; at.n_pages = a->n_pages;
    at.scale = 1.0f / sqrtf((float)D); at.out = w.attn;
    if (tc_attn)
      QD_TRY(launch_prefill_attention_tc(at, w.kv_pack, w.kv_pack_bytes, L), "prefill attention (tcgen05)");
    else
      QD_TRY(launch_prefill_attention(at, L), "prefill attention");
    QD_TRY(proj(l->w.w_o, q8 ? l->w.s_o : nullptr, H, Hq * D, w.attn, EPI_RESID_ADD, w.res), "o gemm");
    QD_TRY(launch_rmsnorm_rows(w.res, l->w.ln_post, n, H, d.rms_eps, w.xn, L), "rmsnorm");
    if ((!q8 || widen) && gemm_tc_swiglu_supported(F, H, n)) {  // SwiGLU in the gate+up GEMM's epilogue
      // h (bf16 [n, F]) goes where the f32 gate/up rows would have gone
      if (widen) {
        QD_TRY(widened(l->w.w_gu, l->w.s_gu, 2 * F, H), "gu widen");
        QD_TRY(launch_gemm_tc_swiglu(w.wide_w, w.xn, F, H, n, w.gu, L_full), "gu swiglu gemm");
      } else {
        QD_TRY(launch_gemm_tc_swiglu(l->w.w_gu, w.xn, F, H, n, w.gu, L), "gu swiglu gemm");
      }
      QD_TRY(proj(l->w.w_down, q8 ? l->w.s_down : nullptr, H, F, w.gu, EPI_RESID_ADD, w.res), "down gemm");
    } else {
      QD_TRY(proj(l->w.w_gu, q8 ? l->w.s_gu : nullptr, 2 * F, H, w.xn, EPI_STORE, w.gu), "gu gemm");
      QD_TRY(launch_swiglu_rows(w.gu, n, F, w.xn, L), "swiglu");
      QD_TRY(proj(l->w.w_down, q8 ? l->w.s_down : nullptr, H, F, w.xn, EPI_RESID_ADD, w.res), "down gemm");
    }
  }
  // the last row alone goes through the final norm, the LM head and the argmax advance
  QD_TRY(launch_rmsnorm_rows(w.res + (size_t)(n - 1) * H, a->final_norm, 1, H, d.rms_eps, w.xn, L), "final rmsnorm");
  QD_TRY(gemm(a->lm_head, a->lm_head_scales, a->vocab, H, w.xn, 1, EPI_STORE, logits), "lm head gemm");
  QD_TRY(launch_prefill_finish(a->pos, n, L), "prefill finish");
  QD_TRY(launch_argmax_advance(logits, a->vocab, 1, a->tok, a->pos, a->step, a->out_tokens, a->max_steps,
                               w.argmax_ws, L),
         "argmax");
  return QD_OK;
}

}  // namespace

size_t qd_verify_workspace_bytes(const qd_step_args* a, int k) {
  if (!a || !a->layers || a->n_layers < 1 || !a->layers[0] || k < 1 || k > kMaxVerify) return 0;
  return verify_ws_layout(a, k, nullptr).total;
}

int qd_verify_step(const qd_step_args* a, const int32_t* draft, int k, float* logits, int32_t* target,
                   int32_t* n_accept, cudaStream_t stream) {
  int rc = validate_verify(a, draft, k, logits, target, n_accept);
  if (rc) return rc;
  return run_verify(a, draft, k, logits, target, n_accept, stream);
}

size_t qd_prefill_workspace_bytes(const qd_step_args* a, int n_tokens) {
  if (!a || !a->layers || a->n_layers < 1 || !a->layers[0] || n_tokens < 1 || n_tokens > kMaxPrefill) return 0;
  return prefill_ws_layout(a, n_tokens, nullptr).total;
}

int qd_prefill(const qd_step_args* a, const int32_t* tokens, int n_tokens, float* logits, cudaStream_t stream) {
  int rc = validate_prefill(a, tokens, n_tokens, logits);
  if (rc) return rc;
  return run_prefill(a, tokens, n_tokens, logits, stream);
}

size_t qd_step_workspace_bytes(const qd_step_args* a) {
  if (!a || !a->layers || a->n_layers < 1 || !a->layers[0] || a->batch < 1) return 0;
  return step_ws_layout(a, nullptr).total;
}

int qd_step_launch_count(const qd_step_args* a) {
  if (!a || a->n_layers < 1 || !a->layers || !a->layers[0]) return 0;
  if (mma_step(a)) return mma_norm_rows() ? 1 + 7 * a->n_layers + 3 : 1 + 5 * a->n_layers + 2;
  if (tc_step(a)) return 1 + 8 * a->n_layers + 3;
  if (a->layers[0]->dims.wtype == QD_W_INT4 || lm_is_w4(a)) return 1 + 5 * a->n_layers + (lm_is_w4(a) ? 1 : 2);
  if (!step_kernels_forced()) {
    std::vector<StreamLayerPtrs> lp;
    StreamStepArgs sa;
    if (stream_args(a, step_ws_layout(a, a->workspace), lp, sa)) return 1;
  }
  return 1 + 5 * a->n_layers + 2;
}

int qd_decode_step(const qd_step_args* a, cudaStream_t stream) {
  int rc = validate_step(a);
  if (rc) return rc;
  return run_step(a, stream);
}

int qd_graph_create(const qd_step_args* a, int steps_per_launch, cudaStream_t stream, qd_graph** out) {
  if (!out) return fail(QD_ERR_INVALID_ARG, "qd_graph_create: null out");
  *out = nullptr;
  if (steps_per_launch < 1 || steps_per_launch > 4096)
    return fail(QD_ERR_INVALID_ARG, "qd_graph_create: steps_per_launch=%d", steps_per_launch);
  int rc = validate_step(a);
  if (rc) return rc;
  if (stream == 0) return fail(QD_ERR_INVALID_ARG, "qd_graph_create: capture needs a non-default stream");
  cudaStreamCaptureStatus st;
  QD_TRY(cudaStreamIsCapturing(stream, &st), "qd_graph_create");
  if (st != cudaStreamCaptureStatusNone) return fail(QD_ERR_INVALID_ARG, "qd_graph_create: stream is capturing");
  QD_TRY(cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal), "begin capture");
  for (int i = 0; i < steps_per_launch; ++i) {
    rc = run_step(a, stream);
    if (rc) {
      cudaGraph_t g;
      cudaStreamEndCapture(stream, &g);
      if (g) cudaGraphDestroy(g);
      return rc;
    }
  }
  cudaGraph_t graph;
  QD_TRY(cudaStreamEndCapture(stream, &graph), "end capture");
  cudaGraphExec_t exec;
  cudaError_t e = cudaGraphInstantiate(&exec, graph, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(graph);
    return cuda_fail(e, "graph instantiate");
  }
  qd_graph* g = new qd_graph;
  g->graph = graph;
  g->exec = exec;
  g->steps = steps_per_launch;
  *out = g;
  return QD_OK;
}

int qd_graph_launch(qd_graph* g, cudaStream_t stream) {
  if (!g) return fail(QD_ERR_INVALID_ARG, "qd_graph_launch: null graph");
  QD_TRY(cudaGraphLaunch(g->exec, stream), "graph launch");
  return QD_OK;
}

int qd_graph_destroy(qd_graph* g) {
  if (!g) return QD_OK;
  cudaGraphExecDestroy(g->exec);
  cudaGraphDestroy(g->graph);
  delete g;
  return QD_OK;
}

int qd_check_device_error(cudaStream_t stream, int* bits) {
  if (!bits) return fail(QD_ERR_INVALID_ARG, "qd_check_device_error: null bits");
  *bits = 0;
  int* p = dev_error_ptr();
  if (!p) return fail(QD_ERR_CUDA, "qd_check_device_error: no device error word");
  int v = 0;
  QD_TRY(cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, stream), "read error word");
  QD_TRY(cudaStreamSynchronize(stream), "sync");
  const int zero = 0;
  QD_TRY(cudaMemcpyAsync(p, &zero, sizeof(int), cudaMemcpyHostToDevice, stream), "clear error word");
  QD_TRY(cudaStreamSynchronize(stream), "sync");
  *bits = v;
  return QD_OK;
}

// ------------------------------------------------------------------ test exports
int qd_debug_q8_block_dots(const int8_t* qs, const void* d_f16, int rows, int cols, const int8_t* x_q,
                           const void* x_d_f16, int32_t* dots, float* y, cudaStream_t stream) {
  if (!qs || !d_f16 || !x_q || !x_d_f16 || !dots || !y || rows < 1 || cols < 32 || cols % 32)
    return fail(QD_ERR_INVALID_ARG, "qd_debug_q8_block_dots: bad arguments");
  if (!gemv_q8_supported(cols)) return fail(QD_ERR_UNSUPPORTED, "qd_debug_q8_block_dots: cols=%d too large", cols);
  if (!aligned16(qs) || !aligned16(x_q) || !aligned16(y) || ((uintptr_t)d_f16 & 1u) || ((uintptr_t)x_d_f16 & 1u))
    return fail(QD_ERR_INVALID_ARG, "qd_debug_q8_block_dots: alignment");
  // the production i8-lane GEMV (the same dispatch as qd_gemv_q8_0), storing its block dots
  GemvQ8Args a = {};
  a.qs = qs; a.d = d_f16; a.R = rows; a.K = cols; a.act = QD_ACT_I8;
  a.pro = PRO_X_F32; a.x = nullptr; a.xq = x_q; a.xd = x_d_f16;
  a.epi = EPI_STORE; a.y = y; a.dots = dots;
  cudaError_t e = launch_gemv_q8(a, make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_debug_q8_block_dots");
}

int qd_debug_paged_indices(const int32_t* page_table, int batch, int max_pages, int page_size, int n_pages,
                           int n_tokens, int32_t* idx, cudaStream_t stream) {
  if (!page_table || !idx || batch < 1 || max_pages < 1 || page_size < 1 || n_pages < 1 || n_tokens < 0 ||
      (long long)n_tokens > (long long)max_pages * page_size)
    return fail(QD_ERR_INVALID_ARG, "qd_debug_paged_indices: bad arguments");
  cudaError_t e = launch_paged_indices(page_table, batch, max_pages, page_size, n_pages, n_tokens, idx,
                                       make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_debug_paged_indices");
}

int qd_debug_wait_timeout(int limit_us, cudaStream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return fail(QD_ERR_INVALID_ARG, "qd_debug_wait_timeout: limit_us=%d", limit_us);
  cudaError_t e = launch_wait_timeout(limit_us, make_launch(stream, false));
  return e == cudaSuccess ? QD_OK : cuda_fail(e, "qd_debug_wait_timeout");
}

}  // extern "C"
