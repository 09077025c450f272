// W4A16 weight-streaming GEMV (batch 1) and the INT4 LM head with a local top-k.
//
// "GPU Kernel Lab" README, "Quantization experiments": a W4A16 decode GEMV and a
// packed INT4 LM head with a local top-k, with per-output-channel weight scales.
// "qwen3-8b-rtx4080-cutedsl" README, "W4A16 dequant-fused GEMM": 4-bit weights halve
// the bytes a decode step streams again, and the dequantisation runs inside the
// streaming loop.
//
// Format: row r holds K codes q in [-8, 7] as offset-binary nibbles u = q + 8, two
// per byte (the even column in the low nibble), and one fp16 scale d[r]:
// w[r, c] = f32(d[r]) * q[r, c]. Activations are bf16 values.
//
// GB300 layout of the work (the batch-1 BF16 ring GEMV's, at a quarter of the
// bytes per weight): one CTA per SM over a contiguous block of rows; a producer
// warp streams the rows through a shared-memory ring with TMA bulk copies (evict-
// first), issued before the programmatic-dependent wait; eight consumer warps own
// fixed 16-byte chunks (32 weights) of every row, their activation slice in
// registers. A nibble becomes the float 1 + u/16 with one shift and one bit
// operation (the nibble placed in the top mantissa bits of 1.0), so a thread's
// chunk sum S = sum (1 + u/16) x over its columns gives sum q x = 16 S - 24 sum x
// exactly up to binary32 rounding (sum x is fixed per thread). Rows reduce through
// a transposed warp butterfly and a fixed-order sum over warps; the epilogue
// scales by d[r].
//
// The LM-head form keeps every row value of the CTA in shared memory, selects the
// CTA's top k (value descending, the lower row first among equal values, NaN never
// chosen), and the last CTA (ticket) merges all candidates in CTA order: the token
// is the first of them (the greedy argmax), and the step's token / position advance
// as in argmax_advance.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <algorithm>
#include <climits>
#include <cstdlib>

namespace qd {
namespace {

constexpr int kConsW = 256;            // consumer threads
constexpr int kRingW = 128 * 1024;     // ring bytes
constexpr int kPhaseW = 128;           // rows reduced per window
constexpr int kMaxTopK = 16;
constexpr int kMaxTopRows = 2048;      // rows of one CTA kept for its top-k

struct W4Params {
  const uint8_t* W;
  const __half* d;
  int R, K;
  int rows_base, rows_extra;
  int T, P, ns, stage_bytes, ring_bytes;
  int pro;
  const void* x;
  const __nv_bfloat16* norm_w;
  float eps;
  int epi;
  float* y;
  __nv_bfloat16* y_bf16;
  int pair_F;
  int w_evict_first;
  int* err;
  int trig_late;
  L2Prefetch pf;
  // EPI_TOPK
  int top_k;
  float* cand_v;
  int* cand_i;
  int* ticket;
  int32_t *tok, *pos, *step, *out_tokens;
  int max_steps;
  int32_t* topk_ids;
  float* topk_vals;
};

QD_DEV void cons_sync_w() { asm volatile("bar.sync 1, %0;" ::"n"(kConsW) : "memory"); }

// sum over the 8 nibbles u_i of one 32-bit word of (1 + u_i / 16) * x[i]; nibble i is
// column i of the word (bytes little-endian, low nibble first)
QD_DEV float dot8_w4(uint32_t w, const float* x) {
  constexpr uint32_t kMask = 0x00780000u, kOne = 0x3F800000u;
  float a = __uint_as_float(((w << 19) & kMask) | kOne) * x[0];
  float b = __uint_as_float(((w << 15) & kMask) | kOne) * x[1];
  a = fmaf(__uint_as_float(((w << 11) & kMask) | kOne), x[2], a);
  b = fmaf(__uint_as_float(((w << 7) & kMask) | kOne), x[3], b);
  a = fmaf(__uint_as_float(((w << 3) & kMask) | kOne), x[4], a);
  b = fmaf(__uint_as_float(((w >> 1) & kMask) | kOne), x[5], b);
  a = fmaf(__uint_as_float(((w >> 5) & kMask) | kOne), x[6], a);
  b = fmaf(__uint_as_float(((w >> 9) & kMask) | kOne), x[7], b);
  return a + b;
}

QD_DEV float silu(float g) { return g / (1.0f + expf(-g)); }

struct Cand {
  float v;
  int i;
};
QD_DEV bool better(const Cand& a, const Cand& b) { return a.v > b.v || (a.v == b.v && a.i < b.i); }

// best candidate of the consumer threads (warp shuffles, then the warps in order);
// sh: [kConsW / 32] scratch; the result is valid in every consumer thread
QD_DEV Cand block_best(Cand c, Cand* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Cand d;
    d.v = __shfl_xor_sync(0xffffffffu, c.v, o);
    d.i = __shfl_xor_sync(0xffffffffu, c.i, o);
    if (better(d, c)) c = d;
  }
  if (lane == 0) sh[warp] = c;
  cons_sync_w();
  Cand b = sh[0];
#pragma unroll
  for (int w = 1; w < kConsW / 32; ++w)
    if (better(sh[w], b)) b = sh[w];
  cons_sync_w();
  return b;
}

template <int C, int RPS>
__global__ void __launch_bounds__(kConsW + 32, 1) gemv_w4_kernel(const W4Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = (uint64_t*)(smem + p.ring_bytes);
  uint64_t* empty = full + 16;
  float* red = (float*)(empty + 16);               // [kPhaseW][wpg]
  float* keep = red + kPhaseW * (kConsW / 32);     // EPI_SWIGLU: [2 npair]; EPI_TOPK: [rows]
  __shared__ float s_ss[kConsW / 32];
  __shared__ Cand s_c[kConsW / 32];
  __shared__ int s_ticket;

  const int tid = threadIdx.x, lane = tid & 31;
  const int K = p.K, ns = p.ns;
  const bool pair = p.epi == EPI_SWIGLU;
  const int nown = p.rows_base + ((int)blockIdx.x < p.rows_extra ? 1 : 0);
  const int npair = pair ? nown : 0;
  const int nrows = pair ? 2 * nown : nown;
  const int r0 = (int)blockIdx.x * p.rows_base + min((int)blockIdx.x, p.rows_extra);
  const int n_stages = (nrows + p.P * RPS - 1) / (p.P * RPS);
  const size_t row_bytes = (size_t)K / 2;

  if (tid == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsW / 32);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (!p.trig_late) pdl_launch_dependents();

  if (tid >= kConsW) {  // ---- producer warp: weights only, so no dependency wait
    if (lane == 0) {
      const unsigned char* src = p.W + (size_t)r0 * row_bytes;
      const unsigned char* src_up = pair ? p.W + ((size_t)p.pair_F + r0) * row_bytes : src;
      const uint64_t pol = policy_evict_first();
      auto copy = [&](void* dd, const void* g, uint32_t n, uint64_t* bar) {
        if (p.w_evict_first) bulk_g2s_hint(dd, g, n, bar, pol);
        else bulk_g2s(dd, g, n, bar);
      };
      for (int i = 0; i < n_stages; ++i) {
        const int slot = i % ns;
        if (i >= ns && !mbar_wait_bounded(&empty[slot], (uint32_t)(((i / ns) - 1) & 1), p.err)) break;
        const int srows = p.P * RPS;
        const int a = i * srows;
        const int rows_i = min(srows, nrows - a);
        mbar_arrive_expect_tx(&full[slot], (uint32_t)(rows_i * row_bytes));
        unsigned char* dst = ring + (size_t)slot * p.stage_bytes;
        if (!pair) {
          copy(dst, src + (size_t)a * row_bytes, (uint32_t)(rows_i * row_bytes), &full[slot]);
        } else {  // the stage may straddle the gate/up boundary: one copy per half
          const int na = max(0, min(a + rows_i, npair) - a);
          if (na > 0) copy(dst, src + (size_t)a * row_bytes, (uint32_t)(na * row_bytes), &full[slot]);
          if (rows_i > na)
            copy(dst + (size_t)na * row_bytes, src_up + (size_t)(a + na - npair) * row_bytes,
                 (uint32_t)((rows_i - na) * row_bytes), &full[slot]);
        }
      }
    }
    __syncwarp();
    pdl_launch_dependents();
    l2_prefetch_spans(p.pf, blockIdx.x, gridDim.x, lane);
    return;
  }

  // ---- consumers: thread t of group g owns 32-column chunks j * T + t of every row
  const int T = p.T, P = p.P;
  const int g = tid / T, t = tid - g * T;
  const int wpg = T >> 5, wig = t >> 5;
  const bool in_grp = g < P;
  int col[C];
  bool cv[C];
#pragma unroll
  for (int j = 0; j < C; ++j) {
    col[j] = (j * T + t) * 32;
    cv[j] = in_grp && col[j] < K;
  }
  uint4 wn[C][4];  // RMSNorm weights of the chunk (loaded before the dependency wait)
#pragma unroll
  for (int j = 0; j < C; ++j)
#pragma unroll
    for (int h = 0; h < 4; ++h)
      wn[j][h] = (p.pro == PRO_RMSNORM && cv[j]) ? *(const uint4*)(p.norm_w + col[j] + 8 * h)
                                                 : make_uint4(0u, 0u, 0u, 0u);
  pdl_wait();

  float x[C][32];
#pragma unroll
  for (int j = 0; j < C; ++j)
#pragma unroll
    for (int e = 0; e < 32; ++e) x[j][e] = 0.f;
  if (p.pro == PRO_X_BF16) {
    const __nv_bfloat16* xb = (const __nv_bfloat16*)p.x;
#pragma unroll
    for (int j = 0; j < C; ++j) {
      if (!cv[j]) continue;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint4 v = *(const uint4*)(xb + col[j] + 8 * h);
        x[j][8 * h + 0] = bf_lo(v.x); x[j][8 * h + 1] = bf_hi(v.x);
        x[j][8 * h + 2] = bf_lo(v.y); x[j][8 * h + 3] = bf_hi(v.y);
        x[j][8 * h + 4] = bf_lo(v.z); x[j][8 * h + 5] = bf_hi(v.z);
        x[j][8 * h + 6] = bf_lo(v.w); x[j][8 * h + 7] = bf_hi(v.w);
      }
    }
  } else {  // PRO_X_F32 or PRO_RMSNORM: f32 source
    const float* xf = (const float*)p.x;
#pragma unroll
    for (int j = 0; j < C; ++j) {
      if (!cv[j]) continue;
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 a = *(const float4*)(xf + col[j] + e);
        x[j][e] = a.x; x[j][e + 1] = a.y; x[j][e + 2] = a.z; x[j][e + 3] = a.w;
      }
    }
    if (p.pro == PRO_X_F32) {
#pragma unroll
      for (int j = 0; j < C; ++j)
#pragma unroll
        for (int e = 0; e < 32; ++e) x[j][e] = round_bf16(x[j][e]);
    } else {
      float ss = 0.f;
      if (g == 0) {
#pragma unroll
        for (int j = 0; j < C; ++j)
#pragma unroll
          for (int e = 0; e < 32; ++e) ss = fmaf(x[j][e], x[j][e], ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) s_ss[tid >> 5] = ss;
      cons_sync_w();
      float tot = 0.f;
      for (int i = 0; i < wpg; ++i) tot += s_ss[i];
      const float inv = 1.0f / sqrtf(tot / (float)K + p.eps);
#pragma unroll
      for (int j = 0; j < C; ++j) {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const uint4 w = wn[j][h];
          const float nw[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y),
                               bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
#pragma unroll
          for (int e = 0; e < 8; ++e)
            x[j][8 * h + e] = cv[j] ? round_bf16(nw[e] * round_bf16(x[j][8 * h + e] * inv)) : 0.f;
        }
      }
    }
  }
  // sum q x = 16 S - 24 sum x over this thread's columns
  float sx = 0.f;
#pragma unroll
  for (int j = 0; j < C; ++j)
#pragma unroll
    for (int e = 0; e < 32; ++e) sx += x[j][e];
  const float corr = 24.0f * sx;

  const bool topk = p.epi == EPI_TOPK;
  Cand best = {-INFINITY, INT_MAX};
  auto epilogue = [&](int lr, float s) {  // lr: local row of the CTA, s: sum q x of it
    if (pair) {
      keep[lr] = s;
      return;
    }
    const int r = r0 + lr;
    const float v = __half2float(p.d[r]) * s;
    if (p.epi == EPI_RESID_ADD) {
      p.y[r] += v;
    } else {
      p.y[r] = v;
      if (topk) keep[lr] = v;
    }
  };

  const int stage_rows = P * RPS;
  int ph_base = 0;
  for (int i = 0; i < n_stages; ++i) {
    const int slot = i % ns;
    if (!mbar_wait_bounded(&full[slot], (uint32_t)((i / ns) & 1), p.err)) {
      for (int k = 1; k < ns && i + k < n_stages; ++k)
        mbar_wait_bounded(&full[(i + k) % ns], (uint32_t)(((i + k) / ns) & 1), p.err);
      return;
    }
    if (i + 1 == n_stages) pdl_launch_dependents();
    const int row0 = i * stage_rows + g * RPS;
    const unsigned char* base = ring + (size_t)slot * p.stage_bytes + (size_t)g * RPS * row_bytes;
    const int nv = in_grp ? min(RPS, nrows - row0) : 0;
    uint4 w[RPS][C];
#pragma unroll
    for (int r = 0; r < RPS; ++r)
#pragma unroll
      for (int j = 0; j < C; ++j)
        w[r][j] = (r < nv && cv[j]) ? *(const uint4*)(base + (size_t)r * row_bytes + (size_t)col[j] / 2)
                                    : make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    float v[RPS];
#pragma unroll
    for (int r = 0; r < RPS; ++r) {
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < C; ++j)
        a += (dot8_w4(w[r][j].x, x[j]) + dot8_w4(w[r][j].y, x[j] + 8)) +
             (dot8_w4(w[r][j].z, x[j] + 16) + dot8_w4(w[r][j].w, x[j] + 24));
      v[r] = 16.0f * a - corr;
    }
    int rsel = 0;
#pragma unroll
    for (int L = 16, n = RPS; L >= 1; L >>= 1) {
      if (n > 1) {
        const int h = n / 2;
        const bool up = (lane & L) != 0;
#pragma unroll
        for (int k = 0; k < h; ++k) {
          const float send = up ? v[k] : v[k + h];
          const float keepv = up ? v[k + h] : v[k];
          v[k] = keepv + __shfl_xor_sync(0xffffffffu, send, L);
        }
        if (up) rsel += h;
        n = h;
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], L);
      }
    }
    constexpr int kLowMask = 32 / RPS - 1;
    if ((lane & kLowMask) == 0 && rsel < nv) red[(row0 + rsel - ph_base) * wpg + wig] = v[0];
    const int done = min((i + 1) * stage_rows, nrows);
    if (done + stage_rows - ph_base > kPhaseW || i + 1 == n_stages) {
      const int nph = done - ph_base;
      cons_sync_w();
      for (int r = tid; r < nph; r += kConsW) {
        float acc = 0.f;
        for (int k = 0; k < wpg; ++k) acc += red[r * wpg + k];
        epilogue(ph_base + r, acc);
      }
      cons_sync_w();
      ph_base = done;
    }
  }
  if (pair) {  // h = bf16(silu(gate) * up) of the CTA's pairs
    for (int j = tid; j < npair; j += kConsW) {
      const float gv = __half2float(p.d[r0 + j]) * keep[j];
      const float uv = __half2float(p.d[p.pair_F + r0 + j]) * keep[npair + j];
      p.y_bf16[r0 + j] = __float2bfloat16_rn(silu(gv) * uv);
    }
    return;
  }
  if (!topk) return;

  // ---- local top-k of the CTA's rows, then the ticket; the last CTA merges
  const int k = p.top_k;
  for (int sel = 0; sel < k; ++sel) {
    Cand c = {-INFINITY, INT_MAX};
    for (int lr = tid; lr < nown; lr += kConsW) {
      const float v = keep[lr];
      if (isnan(v)) continue;
      const Cand d = {v, r0 + lr};
      if (better(d, c)) c = d;
    }
    c = block_best(c, s_c);
    if (tid == 0) {
      p.cand_v[(size_t)blockIdx.x * k + sel] = c.v;
      p.cand_i[(size_t)blockIdx.x * k + sel] = c.i;
      if (c.i != INT_MAX) keep[c.i - r0] = __int_as_float(0x7fffffff);  // taken: NaN from now on
    }
    cons_sync_w();
  }
  if (tid == 0) {
    __threadfence();
    s_ticket = atomicAdd(p.ticket, 1);
  }
  cons_sync_w();
  if (s_ticket != (int)gridDim.x - 1) return;
  __threadfence();
  const int nc = (int)gridDim.x * k;
  float* cv_ = keep;                 // the candidates' values, NaN once taken
  int* ci_ = (int*)(keep + nc);      // and their rows
  for (int e = tid; e < nc; e += kConsW) {
    cv_[e] = __ldcg(p.cand_v + e);
    ci_[e] = __ldcg(p.cand_i + e);
  }
  cons_sync_w();
  int first = INT_MAX;
  for (int sel = 0; sel < k; ++sel) {
    Cand c = {-INFINITY, INT_MAX};
    for (int e = tid; e < nc; e += kConsW) {
      const Cand d = {cv_[e], ci_[e]};
      if (!isnan(d.v) && d.i != INT_MAX && better(d, c)) c = d;
    }
    c = block_best(c, s_c);   // every row is a candidate of one CTA at most
    for (int e = tid; e < nc; e += kConsW)
      if (c.i != INT_MAX && ci_[e] == c.i) cv_[e] = __int_as_float(0x7fffffff);
    if (tid == 0) {
      if (p.topk_ids) p.topk_ids[sel] = c.i == INT_MAX ? -1 : c.i;
      if (p.topk_vals) p.topk_vals[sel] = c.v;
      if (sel == 0) first = c.i;
    }
    cons_sync_w();
  }
  if (tid == 0) {
    int tk = first;
    if (tk == INT_MAX) {
      set_error(p.err, QD_DEVERR_NAN);
      tk = 0;
    }
    if (p.tok) {
      const int st = p.step[0];
      if (st >= 0 && st < p.max_steps) p.out_tokens[st] = tk;
      else set_error(p.err, QD_DEVERR_STEPS);
      p.tok[0] = tk;
      p.pos[0] += 1;
      p.step[0] = st + 1;
    }
    *p.ticket = 0;
  }
}

int w4_c(int K) {  // 32-column chunks per thread (K <= 16384)
  const int chunks = K / 32;
  return chunks <= kConsW ? 1 : chunks <= 2 * kConsW ? 2 : 0;
}

template <int C>
cudaError_t launch_w4_c(const W4Params& p, int grid, size_t smem, const Launch& L) {
  constexpr int RPS = C == 1 ? 8 : 4;
  auto k = gemv_w4_kernel<C, RPS>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dev_info().max_smem_optin - 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(k, dim3(grid), dim3(kConsW + 32), smem, L, p);
}

}  // namespace

bool gemv_w4_supported(int K) { return K >= 32 && K % 32 == 0 && w4_c(K) > 0; }

// candidates [SMs][kMaxTopK] (value, row) and the merge ticket
size_t w4_topk_workspace_bytes() {
  return (((size_t)dev_info().sm_count * kMaxTopK * 8 + 255) & ~(size_t)255) + 256;
}

cudaError_t launch_gemv_w4(const GemvW4Args& a, const Launch& L) {
  const int rc = w4_c(a.K);
  if (rc == 0 || a.K % 32) return cudaErrorInvalidValue;
  const bool pair = a.epi == EPI_SWIGLU, topk = a.epi == EPI_TOPK;
  if (topk && (a.top_k < 1 || a.top_k > kMaxTopK || !a.ws)) return cudaErrorInvalidValue;
  W4Params p = {};
  p.W = (const uint8_t*)a.W;
  p.d = (const __half*)a.d;
  p.R = a.R; p.K = a.K;
  const int units = pair ? a.R / 2 : a.R;
  const int grid = std::max(1, std::min(units, dev_info().sm_count));
  p.rows_base = units / grid; p.rows_extra = units % grid;
  if (topk && p.rows_base + 1 > kMaxTopRows) return cudaErrorInvalidValue;
  p.pair_F = pair ? a.R / 2 : 0;
  const int chunks = a.K / 32;
  p.T = std::min(kConsW, ((ceil_div(chunks, rc) + 31) / 32) * 32);
  p.P = std::max(1, kConsW / p.T);
  const int rps = rc == 1 ? 8 : 4;   // must match launch_w4_c
  const int row_bytes = a.K / 2;
  p.stage_bytes = ((p.P * rps * row_bytes + 127) / 128) * 128;
  p.ns = std::max(2, std::min(16, kRingW / p.stage_bytes));
  p.ring_bytes = p.ns * p.stage_bytes;
  p.pro = a.pro; p.x = a.x; p.norm_w = (const __nv_bfloat16*)a.norm_w; p.eps = a.eps;
  p.epi = a.epi; p.y = a.y; p.y_bf16 = (__nv_bfloat16*)a.y_bf16;
  p.w_evict_first = a.w_evict_first;
  p.err = L.err; p.trig_late = L.trig_late;
  p.pf = a.pf;
  if (topk) {
    unsigned char* ws = (unsigned char*)a.ws;
    const size_t cb = (((size_t)dev_info().sm_count * kMaxTopK * 8 + 255) & ~(size_t)255);
    p.top_k = a.top_k;
    p.cand_v = (float*)ws;
    p.cand_i = (int*)(ws + (size_t)dev_info().sm_count * kMaxTopK * 4);
    p.ticket = (int*)(ws + cb);
    p.tok = a.tok; p.pos = a.pos; p.step = a.step; p.out_tokens = a.out_tokens; p.max_steps = a.max_steps;
    p.topk_ids = a.topk_ids; p.topk_vals = a.topk_vals;
  }
  size_t keep_floats = pair ? 2 * (size_t)(p.rows_base + 1)
                      : topk ? std::max((size_t)(p.rows_base + 1), (size_t)2 * grid * a.top_k) : 0;
  size_t smem = (size_t)p.ring_bytes + 32 * 8 + (size_t)kPhaseW * (kConsW / 32) * 4 + keep_floats * 4;
  if (smem > (size_t)dev_info().max_smem_optin - 2048) return cudaErrorInvalidValue;
  smem = std::max(smem, (size_t)dev_info().max_smem_optin / 2 + 1024);  // one GEMV CTA per SM
  return rc == 1 ? launch_w4_c<1>(p, grid, smem, L) : launch_w4_c<2>(p, grid, smem, L);
}

}  // namespace qd
