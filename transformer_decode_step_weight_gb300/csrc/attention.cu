// GQA split-KV decode attention over a paged bf16 KV cache, with the per-head
// QK RMSNorm, RoPE and the K/V cache write of the current token fused in.
//
// "qwen3-8b-rtx4080-cutedsl" README, "Split-KV decode attention": the sequence
// is split across CTAs (Flash-Decoding) and a final pass combines the partial
// softmax states; the q heads that share a KV head are packed into one CTA.
// Same README, "GQA + QK-Norm": kv head = q head / (Hq / Hkv); per-head RMSNorm
// of q and k before the scores. "GPU Kernel Lab" README, "Decode integration":
// Q/K RMSNorm + RoPE + direct K/V cache write, then split-KV online-softmax
// attention; "Measured final results": K/V in fixed physical pages read
// through a page table.
//
// GB300 design:
//   * grid (split, kv head, sequence), 128 threads; each CTA owns 64 tokens of
//     one kv head and all REP = Hq/Hkv q heads that read it;
//   * one thread issues TMA bulk copies (cp.async.bulk, 256 B per token row,
//     one copy per contiguous page segment) of the chunk's K and V into shared
//     memory on an mbarrier while the CTA computes q (and the new k, v);
//   * scores, softmax and P.V run from shared memory in f32; a split writes
//     (m, l, acc[REP][128]) to the workspace and takes a ticket; the last split
//     of a (sequence, kv head) combines all partials in split order (fixed, so
//     the result is deterministic) and resets the ticket to zero. No spin-wait.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace qd {
namespace {

constexpr int kD = 128;
constexpr int kChunk = 64;
constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  const float* q;
  const float* qkv;
  const __nv_bfloat16* q_norm;
  const __nv_bfloat16* k_norm;
  const float2* rope;
  int rope_max_pos;
  float eps;
  const int32_t* pos;
  const int32_t* seq_lens;
  __nv_bfloat16* k_pages;
  __nv_bfloat16* v_pages;
  const int32_t* page_table;
  int B, Hq, Hkv, page_size, max_pages, n_pages, n_splits;
  float scale_log2;
  float* out_f32;
  __nv_bfloat16* out_bf16;
  float* ws_acc;
  float* ws_ml;
  int* ws_cnt;
  int* err;
};

struct Carve {
  size_t k, v, q, s, ml, bar, total;
};
__host__ __device__ inline Carve carve(int rep) {
  Carve c;
  c.k = 0;
  c.v = c.k + kChunk * kD * 2;
  c.q = c.v + kChunk * kD * 2;
  c.s = c.q + (size_t)rep * kD * 4;
  c.ml = c.s + (size_t)rep * kChunk * 4;
  c.bar = c.ml + 64 * 4;
  c.total = c.bar + 16;
  return c;
}

// Per-head RMSNorm (Qwen cast order) + RoPE of one 128-vector held one element
// per thread; returns this thread's rotated element (f32). `red` holds 4 floats.
QD_DEV float norm_rope(float x, const __nv_bfloat16* w, const float2* rope_row, float eps,
                       float* red, float* xs) {
  const int d = threadIdx.x;
  float ss = warp_sum(x * x);
  if ((d & 31) == 0) red[d >> 5] = ss;
  __syncthreads();
  ss = (red[0] + red[1]) + (red[2] + red[3]);
  const float inv = 1.0f / sqrtf(ss / (float)kD + eps);
  const float y = round_bf16(__bfloat162float(w[d]) * round_bf16(x * inv));
  xs[d] = y;
  __syncthreads();
  const int j = d & 63;
  const float2 cs = rope_row[j];
  const float other = xs[d ^ 64];
  const float r = (d < 64) ? (y * cs.x - other * cs.y) : (y * cs.x + other * cs.y);
  __syncthreads();  // xs and red are reused by the next call
  return r;
}

template <int REP, bool FUSED>
__global__ void __launch_bounds__(kThreads) attn_kernel(const AttnParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const Carve cv = carve(REP);
  __nv_bfloat16* sK = (__nv_bfloat16*)(smem + cv.k);
  __nv_bfloat16* sV = (__nv_bfloat16*)(smem + cv.v);
  float* sQ = (float*)(smem + cv.q);
  float* sS = (float*)(smem + cv.s);
  float* sML = (float*)(smem + cv.ml);  // [0..REP) m, [REP..2REP) l, [32..36) scratch
  uint64_t* bar = (uint64_t*)(smem + cv.bar);
  __shared__ int s_ticket;
  __shared__ float s_x[kD];

  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  pdl_wait();
  pdl_launch_dependents();

  int len, pos = 0;
  if (FUSED) {
    pos = p.pos[b];
    len = pos + 1;
  } else {
    len = p.seq_lens[b];
  }
  const int cap = p.max_pages * p.page_size;
  if (len < 0 || len > cap || (FUSED && (pos < 0 || pos >= p.rope_max_pos))) {
    if (s == 0 && tid == 0) set_error(p.err, QD_DEVERR_POS);
    return;
  }
  const int n_act = (len + kChunk - 1) / kChunk;
  if (len == 0) {  // empty sequence: zero output (standalone form only)
    if (s == 0 && !FUSED)
      for (int i = 0; i < REP; ++i)
        p.out_f32[((size_t)b * p.Hq + g * REP + i) * kD + tid] = 0.f;
    return;
  }
  if (s >= n_act) return;

  const int t0 = s * kChunk;
  const int nv = min(kChunk, len - t0);
  const int ncopy = FUSED ? min(nv, pos - t0) : nv;
  const int ps = p.page_size;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, (uint32_t)ncopy * kD * 2 * 2);
    const int32_t* pt = p.page_table + (size_t)b * p.max_pages;
    int t = t0;
    const int end = t0 + ncopy;
    while (t < end) {
      const int lp = t / ps;
      int page = pt[lp];
      if (page < 0 || page >= p.n_pages) {
        set_error(p.err, QD_DEVERR_PAGE);
        page = 0;
      }
      const int seg_end = min(end, (lp + 1) * ps);
      const size_t off = (((size_t)page * p.Hkv + g) * ps + (t - lp * ps)) * kD;
      const uint32_t bytes = (uint32_t)(seg_end - t) * kD * 2;
      bulk_g2s(sK + (size_t)(t - t0) * kD, p.k_pages + off, bytes, bar);
      bulk_g2s(sV + (size_t)(t - t0) * kD, p.v_pages + off, bytes, bar);
      t = seg_end;
    }
  }

  // ---- q for the REP heads of this kv head (pre-scaled by scale * log2 e)
  if (FUSED) {
    const int qkv_w = (p.Hq + 2 * p.Hkv) * kD;
    const float* qkv = p.qkv + (size_t)b * qkv_w;
    const float2* rope_row = p.rope + (size_t)pos * (kD / 2);
#pragma unroll 1
    for (int i = 0; i < REP; ++i) {
      const float x = qkv[(g * REP + i) * kD + tid];
      const float r = norm_rope(x, p.q_norm, rope_row, p.eps, sML + 32, s_x);
      sQ[i * kD + tid] = r * p.scale_log2;
    }
    if (pos < t0 + kChunk) {  // this split holds the current token: build and store k, v
      const float kx = qkv[(p.Hq + g) * kD + tid];
      const float kr = round_bf16(norm_rope(kx, p.k_norm, rope_row, p.eps, sML + 32, s_x));
      const float vr = round_bf16(qkv[(p.Hq + p.Hkv + g) * kD + tid]);
      const int lp = pos / ps;
      int page = p.page_table[(size_t)b * p.max_pages + lp];
      if (page < 0 || page >= p.n_pages) {
        if (tid == 0) set_error(p.err, QD_DEVERR_PAGE);
      } else {
        const size_t off = (((size_t)page * p.Hkv + g) * ps + (pos - lp * ps)) * kD + tid;
        p.k_pages[off] = __float2bfloat16_rn(kr);
        p.v_pages[off] = __float2bfloat16_rn(vr);
      }
      sK[(size_t)(pos - t0) * kD + tid] = __float2bfloat16_rn(kr);
      sV[(size_t)(pos - t0) * kD + tid] = __float2bfloat16_rn(vr);
    }
  } else {
#pragma unroll
    for (int i = 0; i < REP; ++i)
      sQ[i * kD + tid] = p.q[((size_t)b * p.Hq + g * REP + i) * kD + tid] * p.scale_log2;
  }
  __syncthreads();
  if (!mbar_wait_bounded(bar, 0, p.err)) {
    mbar_wait_bounded(bar, 0, p.err);  // give copies in flight a second bounded chance
    return;
  }

  // ---- scores: lane = (token half, 16-byte dim chunk); warp w owns pairs [8w, 8w + 8)
  const int half = lane >> 4, dc = lane & 15;
  float qr[REP][8];
#pragma unroll
  for (int i = 0; i < REP; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) qr[i][e] = sQ[i * kD + dc * 8 + e];

#pragma unroll 2
  for (int pi = warp * 8; pi < warp * 8 + 8; ++pi) {
    const int tt = 2 * pi + half;
    const bool ok = tt < nv;
    uint4 kw = make_uint4(0u, 0u, 0u, 0u);
    if (ok) kw = *(const uint4*)(sK + (size_t)tt * kD + dc * 8);
    const float kf[8] = {bf_lo(kw.x), bf_hi(kw.x), bf_lo(kw.y), bf_hi(kw.y),
                         bf_lo(kw.z), bf_hi(kw.z), bf_lo(kw.w), bf_hi(kw.w)};
#pragma unroll
    for (int i = 0; i < REP; ++i) {
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) a = fmaf(kf[e], qr[i][e], a);
      a += __shfl_xor_sync(0xffffffffu, a, 8);
      a += __shfl_xor_sync(0xffffffffu, a, 4);
      a += __shfl_xor_sync(0xffffffffu, a, 2);
      a += __shfl_xor_sync(0xffffffffu, a, 1);
      if (dc == 0) sS[i * kChunk + tt] = ok ? a : -INFINITY;
    }
  }
  __syncthreads();

  // ---- chunk softmax per head (log2 domain)
  for (int i = warp; i < REP; i += kThreads / 32) {
    const float a0 = sS[i * kChunk + lane], a1 = sS[i * kChunk + lane + 32];
    const float m = warp_max(fmaxf(a0, a1));
    const float e0 = exp2f(a0 - m), e1 = exp2f(a1 - m);
    const float l = warp_sum(e0 + e1);
    sS[i * kChunk + lane] = e0;
    sS[i * kChunk + lane + 32] = e1;
    if (lane == 0) {
      sML[i] = m;
      sML[REP + i] = l;
    }
  }
  __syncthreads();

  // ---- P . V
  float acc[REP][8];
#pragma unroll
  for (int i = 0; i < REP; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
#pragma unroll 2
  for (int pi = warp * 8; pi < warp * 8 + 8; ++pi) {
    const int tt = 2 * pi + half;
    if (tt < nv) {
      const uint4 vw = *(const uint4*)(sV + (size_t)tt * kD + dc * 8);
      const float vf[8] = {bf_lo(vw.x), bf_hi(vw.x), bf_lo(vw.y), bf_hi(vw.y),
                           bf_lo(vw.z), bf_hi(vw.z), bf_lo(vw.w), bf_hi(vw.w)};
#pragma unroll
      for (int i = 0; i < REP; ++i) {
        const float pp = sS[i * kChunk + tt];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(pp, vf[e], acc[i][e]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < REP; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] += __shfl_xor_sync(0xffffffffu, acc[i][e], 16);
  float* sRed = (float*)sK;  // K tile no longer needed: [4 warps][REP][128]
  if (half == 0) {
#pragma unroll
    for (int i = 0; i < REP; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) sRed[(warp * REP + i) * kD + dc * 8 + e] = acc[i][e];
  }
  __syncthreads();
  float o[REP];
#pragma unroll
  for (int i = 0; i < REP; ++i)
    o[i] = (sRed[(0 * REP + i) * kD + tid] + sRed[(1 * REP + i) * kD + tid]) +
           (sRed[(2 * REP + i) * kD + tid] + sRed[(3 * REP + i) * kD + tid]);

  const size_t head0 = (size_t)b * p.Hq + g * REP;
  if (n_act == 1) {  // a single split is already complete
#pragma unroll
    for (int i = 0; i < REP; ++i) {
      const float r = o[i] / sML[REP + i];
      if (p.out_bf16) p.out_bf16[(head0 + i) * kD + tid] = __float2bfloat16_rn(r);
      else p.out_f32[(head0 + i) * kD + tid] = r;
    }
    return;
  }

  // ---- publish the partial, take a ticket; the last split combines
  const size_t slot = ((size_t)b * p.Hkv + g) * p.n_splits + s;
#pragma unroll
  for (int i = 0; i < REP; ++i) p.ws_acc[(slot * REP + i) * kD + tid] = o[i];
  if (tid < REP) {
    p.ws_ml[(slot * REP + tid) * 2 + 0] = sML[tid];
    p.ws_ml[(slot * REP + tid) * 2 + 1] = sML[REP + tid];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_ticket = atomicAdd(p.ws_cnt + (size_t)b * p.Hkv + g, 1);
  __syncthreads();
  if (s_ticket != n_act - 1) return;
  __threadfence();

  const size_t slot0 = ((size_t)b * p.Hkv + g) * p.n_splits;
#pragma unroll 1
  for (int i = 0; i < REP; ++i) {
    float M = -INFINITY;
    for (int k = 0; k < n_act; ++k) M = fmaxf(M, __ldcg(p.ws_ml + ((slot0 + k) * REP + i) * 2));
    float L = 0.f, O = 0.f;
    for (int k = 0; k < n_act; ++k) {
      const float m = __ldcg(p.ws_ml + ((slot0 + k) * REP + i) * 2);
      const float l = __ldcg(p.ws_ml + ((slot0 + k) * REP + i) * 2 + 1);
      const float w = exp2f(m - M);
      L = fmaf(w, l, L);
      O = fmaf(w, __ldcg(p.ws_acc + ((slot0 + k) * REP + i) * kD + tid), O);
    }
    const float r = O / L;
    if (p.out_bf16) p.out_bf16[(head0 + i) * kD + tid] = __float2bfloat16_rn(r);
    else p.out_f32[(head0 + i) * kD + tid] = r;
  }
  if (tid == 0) p.ws_cnt[(size_t)b * p.Hkv + g] = 0;
}

__global__ void rope_table_kernel(float2* table, int max_pos, int half, double theta) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)max_pos * half) return;
  const int p = (int)(i / half), j = (int)(i % half);
  const double inv = pow(theta, -2.0 * (double)j / (double)(2 * half));
  double sn, cs;
  sincos((double)p * inv, &sn, &cs);
  table[i] = make_float2((float)cs, (float)sn);
}

template <int REP, bool FUSED>
cudaError_t launch_rep(const AttnParams& prm, const Launch& L) {
  auto k = attn_kernel<REP, FUSED>;
  const size_t smem = carve(REP).total;
  dim3 grid(prm.n_splits, prm.Hkv, prm.B);
  return launch_ex(k, grid, dim3(kThreads), smem, L, prm);
}

}  // namespace

size_t attn_workspace_bytes(int B, int Hq, int Hkv, int max_ctx) {
  const int rep = Hq / Hkv;
  const size_t splits = (size_t)(max_ctx + kChunk - 1) / kChunk;
  const size_t slots = (size_t)B * Hkv * splits;
  size_t acc = slots * rep * kD * 4;
  size_t ml = slots * rep * 2 * 4;
  size_t cnt = (size_t)B * Hkv * 4;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al(acc) + al(ml) + al(cnt);
}

cudaError_t launch_attention(const AttnArgs& a, const Launch& L) {
  AttnParams p;
  const int rep = a.Hq / a.Hkv;
  p.q = a.q;
  p.qkv = a.qkv;
  p.q_norm = (const __nv_bfloat16*)a.q_norm;
  p.k_norm = (const __nv_bfloat16*)a.k_norm;
  p.rope = (const float2*)a.rope;
  p.rope_max_pos = a.rope_max_pos;
  p.eps = a.eps;
  p.pos = a.pos;
  p.seq_lens = a.seq_lens;
  p.k_pages = (__nv_bfloat16*)a.k_pages;
  p.v_pages = (__nv_bfloat16*)a.v_pages;
  p.page_table = a.page_table;
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv;
  p.page_size = a.page_size; p.max_pages = a.max_pages; p.n_pages = a.n_pages;
  p.n_splits = (a.max_ctx + kChunk - 1) / kChunk;
  p.scale_log2 = a.scale * kLog2e;
  p.out_f32 = a.out_f32;
  p.out_bf16 = (__nv_bfloat16*)a.out_bf16;
  const size_t slots = (size_t)a.B * a.Hkv * p.n_splits;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  unsigned char* ws = (unsigned char*)a.workspace;
  p.ws_acc = (float*)ws;
  p.ws_ml = (float*)(ws + al(slots * rep * kD * 4));
  p.ws_cnt = (int*)(ws + al(slots * rep * kD * 4) + al(slots * rep * 2 * 4));
  p.err = L.err;
  const bool fused = a.qkv != nullptr;
#define QD_ATTN_CASE(R)                                                      \
  case R:                                                                    \
    return fused ? launch_rep<R, true>(p, L) : launch_rep<R, false>(p, L);
  switch (rep) {
    QD_ATTN_CASE(1)
    QD_ATTN_CASE(2)
    QD_ATTN_CASE(4)
    QD_ATTN_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef QD_ATTN_CASE
}

cudaError_t launch_rope_table(float* table, int max_pos, int head_dim, float theta, cudaStream_t s) {
  const int half = head_dim / 2;
  const long long n = (long long)max_pos * half;
  const int threads = 256;
  const int blocks = (int)((n + threads - 1) / threads);
  rope_table_kernel<<<blocks, threads, 0, s>>>((float2*)table, max_pos, half, (double)theta);
  return cudaGetLastError();
}

}  // namespace qd
