// Embedding gather, greedy argmax with on-device token/position advance, and
// the paged-index debug export.
//
// "GPU Kernel Lab" README, "Decode integration": fixed token/position buffers
// feed the step, and the LM-head GEMV is followed by argmax + token/position
// update on the device. "emit_qwen38_generate" rustdoc, "Where the speed comes
// from", item 2: the sampled token and the position advance ON DEVICE so no
// graph replay needs a host round trip.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <climits>

namespace qd {
namespace {

constexpr int kArgmaxBlocks = 32;
constexpr int kArgmaxThreads = 512;

// res[b, :] = f32(embed[tok[b], :])
__global__ void __launch_bounds__(256) embed_kernel(const __nv_bfloat16* embed, int H, int V,
                                                    const int32_t* tok, float* res, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.y;
  int t = tok[b];
  if (t < 0 || t >= V) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_error(err, QD_DEVERR_PAGE);
    t = 0;
  }
  const __nv_bfloat16* row = embed + (size_t)t * H;
  for (int i = (blockIdx.x * blockDim.x + threadIdx.x) * 8; i < H; i += gridDim.x * blockDim.x * 8) {
    const uint4 v = *(const uint4*)(row + i);
    float4 a = make_float4(bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y));
    float4 c = make_float4(bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w));
    *(float4*)(res + (size_t)b * H + i) = a;
    *(float4*)(res + (size_t)b * H + i + 4) = c;
  }
}

// (value, index) candidates; NaN maps to (-inf, INT_MAX) so it never wins and
// an all-NaN row is recognisable.
struct Cand {
  float v;
  int i;
};
QD_DEV bool better(const Cand& a, const Cand& b) { return a.v > b.v || (a.v == b.v && a.i < b.i); }

QD_DEV Cand block_argmax(Cand c, Cand* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Cand d;
    d.v = __shfl_xor_sync(0xffffffffu, c.v, o);
    d.i = __shfl_xor_sync(0xffffffffu, c.i, o);
    if (better(d, c)) c = d;
  }
  if (lane == 0) sh[warp] = c;
  __syncthreads();
  if (warp == 0) {
    c = lane < (int)(blockDim.x >> 5) ? sh[lane] : Cand{-INFINITY, INT_MAX};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Cand d;
      d.v = __shfl_xor_sync(0xffffffffu, c.v, o);
      d.i = __shfl_xor_sync(0xffffffffu, c.i, o);
      if (better(d, c)) c = d;
    }
  }
  return c;  // valid in warp 0
}

struct ArgmaxParams {
  const float* logits;
  int V, B;
  int32_t *tok, *pos, *step, *out;
  int max_steps;
  Cand* cand;  // [B, kArgmaxBlocks]
  int* cnt;    // [B]
  int* err;
};

__global__ void __launch_bounds__(kArgmaxThreads) argmax_advance_kernel(const ArgmaxParams p) {
  __shared__ Cand sh[32];
  __shared__ int s_ticket;
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.y;
  const float* row = p.logits + (size_t)b * p.V;
  const int per = (p.V + gridDim.x - 1) / gridDim.x;
  const int lo = blockIdx.x * per, hi = min(p.V, lo + per);
  Cand c{-INFINITY, INT_MAX};
  for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    const float v = row[i];
    Cand d{isnan(v) ? -INFINITY : v, isnan(v) ? INT_MAX : i};
    if (better(d, c)) c = d;
  }
  c = block_argmax(c, sh);
  if (threadIdx.x == 0) {
    p.cand[b * gridDim.x + blockIdx.x] = c;
    __threadfence();
    s_ticket = atomicAdd(p.cnt + b, 1);
  }
  __syncthreads();
  if (s_ticket != (int)gridDim.x - 1) return;
  __threadfence();
  // last block of this row: reduce the candidates in block order
  if (threadIdx.x == 0) {
    Cand best{-INFINITY, INT_MAX};
    for (int k = 0; k < (int)gridDim.x; ++k) {
      Cand d;
      d.v = __ldcg(&p.cand[b * gridDim.x + k].v);
      d.i = __ldcg(&p.cand[b * gridDim.x + k].i);
      if (better(d, best)) best = d;
    }
    int t = best.i;
    if (t == INT_MAX) {
      set_error(p.err, QD_DEVERR_NAN);
      t = 0;
    }
    const int st = p.step[b];
    if (st >= 0 && st < p.max_steps) p.out[(size_t)b * p.max_steps + st] = t;
    else set_error(p.err, QD_DEVERR_STEPS);
    p.tok[b] = t;
    p.pos[b] += 1;
    p.step[b] = st + 1;
    p.cnt[b] = 0;
  }
}

// out[b, :] = bf16(w * bf16(x[b, :] * rsqrt(mean(x[b, :]^2) + eps))), Qwen cast order.
// One CTA per row; each thread keeps CPT 8-element chunks of the row in registers
// (one pass over x), the weights are loaded before the dependency wait.
template <int CPT>
__global__ void __launch_bounds__(256) rmsnorm_rows_kernel(const float* x, const __nv_bfloat16* w, int K, float eps,
                                                           __nv_bfloat16* out) {
  __shared__ float red[8];
  const int b = blockIdx.x, tid = threadIdx.x;
  uint4 wv[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    const int i = (c * 256 + tid) * 8;
    wv[c] = i < K ? *(const uint4*)(w + i) : make_uint4(0u, 0u, 0u, 0u);
  }
  pdl_wait();
  pdl_launch_dependents();
  const float* xr = x + (size_t)b * K;
  float xv[CPT][8];
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    const int i = (c * 256 + tid) * 8;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), d = a;
    if (i < K) {
      a = *(const float4*)(xr + i);
      d = *(const float4*)(xr + i + 4);
    }
    xv[c][0] = a.x; xv[c][1] = a.y; xv[c][2] = a.z; xv[c][3] = a.w;
    xv[c][4] = d.x; xv[c][5] = d.y; xv[c][6] = d.z; xv[c][7] = d.w;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(xv[c][e], xv[c][e], ss);
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += red[i];
  const float inv = 1.0f / sqrtf(tot / (float)K + eps);
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    const int i = (c * 256 + tid) * 8;
    if (i >= K) continue;
    const float wf[8] = {bf_lo(wv[c].x), bf_hi(wv[c].x), bf_lo(wv[c].y), bf_hi(wv[c].y),
                         bf_lo(wv[c].z), bf_hi(wv[c].z), bf_lo(wv[c].w), bf_hi(wv[c].w)};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat16 lo = __float2bfloat16_rn(wf[2 * e] * round_bf16(xv[c][2 * e] * inv));
      const __nv_bfloat16 hi = __float2bfloat16_rn(wf[2 * e + 1] * round_bf16(xv[c][2 * e + 1] * inv));
      o[e] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
    }
    *(uint4*)(out + (size_t)b * K + i) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// out[b, j] = bf16(silu(g) * u) with g = gu[b, j], u = gu[b, F + j]
__global__ void __launch_bounds__(256) swiglu_rows_kernel(const float* gu, int F, __nv_bfloat16* out) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.y;
  const float* row = gu + (size_t)b * 2 * F;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < F; j += gridDim.x * blockDim.x) {
    const float g = row[j], u = row[F + j];
    out[(size_t)b * F + j] = __float2bfloat16_rn(g / (1.0f + expf(-g)) * u);
  }
}

// The physical token slot of logical token t, through the attention kernels' own
// page-table lookup (paged_slot); -1 and QD_DEVERR_PAGE for an id out of range.
__global__ void paged_indices_kernel(const int32_t* pt, int B, int max_pages, int ps, int n_pages, int n,
                                     int32_t* idx, int* err) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)B * n) return;
  const int b = (int)(i / n), t = (int)(i % n);
  const PagedSlot sl = paged_slot(pt + (size_t)b * max_pages, t, ps, n_pages);
  if (!sl.ok) set_error(err, QD_DEVERR_PAGE);
  idx[i] = sl.ok ? sl.page * ps + sl.slot : -1;
}

// Row inputs of a speculative verify pass (one sequence, k rows).
__global__ void verify_prep_kernel(const int32_t* tok, const int32_t* pos, const int32_t* draft, int k,
                                   const int32_t* page_table, int max_pages, int32_t* tokens, int32_t* vpos,
                                   int32_t* vpt, int32_t* scratch) {
  pdl_wait();
  pdl_launch_dependents();
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    tokens[i] = i == 0 ? tok[0] : draft[i - 1];
    vpos[i] = pos[0] + i;
    scratch[i] = 0;             // argmax scratch: position
    scratch[k + i] = 0;         // ... and step (one output slot per row)
  }
  for (int e = threadIdx.x; e < k * max_pages; e += blockDim.x) vpt[e] = page_table[e % max_pages];
}

// The accepted prefix of the drafts and the state advance (one thread).
__global__ void verify_accept_kernel(const int32_t* draft, const int32_t* target, int k, int32_t* tok, int32_t* pos,
                                     int32_t* step, int32_t* out_tokens, int max_steps, int32_t* n_accept, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x != 0) return;
  int m = 0;
  while (m < k - 1 && draft[m] == target[m]) ++m;
  const int st = step[0];
  for (int i = 0; i <= m; ++i) {
    const int t = i < m ? draft[i] : target[m];
    if (st + i >= 0 && st + i < max_steps) out_tokens[st + i] = t;
    else set_error(err, QD_DEVERR_STEPS);
  }
  tok[0] = target[m];
  pos[0] += m + 1;
  step[0] = st + m + 1;
  n_accept[0] = m;
}

}  // namespace

// A wait that runs out: one thread arms an mbarrier for 16 bytes that no copy will
// ever deliver (nothing is issued, so nothing is in flight), then waits on it with a
// limit of limit_us microseconds; the wait gives up, sets QD_DEVERR_TIMEOUT and the
// kernel returns.
__global__ void wait_timeout_kernel(int limit_us, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_arrive_expect_tx(&bar, 16);
  mbar_wait_limit(&bar, 0, err, (uint64_t)limit_us * 1000ull);
}

cudaError_t launch_wait_timeout(int limit_us, const Launch& L) {
  return launch_ex(wait_timeout_kernel, dim3(1), dim3(32), 0, L, limit_us, L.err);
}

cudaError_t launch_verify_prep(const int32_t* tok, const int32_t* pos, const int32_t* draft, int k,
                               const int32_t* page_table, int max_pages, int32_t* tokens, int32_t* vpos,
                               int32_t* vpt, int32_t* scratch, const Launch& L) {
  return launch_ex(verify_prep_kernel, dim3(1), dim3(256), 0, L, tok, pos, draft, k, page_table, max_pages, tokens,
                   vpos, vpt, scratch);
}

cudaError_t launch_verify_accept(const int32_t* draft, const int32_t* target, int k, int32_t* tok, int32_t* pos,
                                 int32_t* step, int32_t* out_tokens, int max_steps, int32_t* n_accept,
                                 const Launch& L) {
  return launch_ex(verify_accept_kernel, dim3(1), dim3(32), 0, L, draft, target, k, tok, pos, step, out_tokens,
                   max_steps, n_accept, L.err);
}

size_t argmax_workspace_bytes(int B) {
  return (((size_t)B * kArgmaxBlocks * sizeof(Cand) + 255) & ~(size_t)255) + (size_t)B * 4;
}

cudaError_t launch_argmax_advance(const float* logits, int V, int B, int32_t* tok, int32_t* pos,
                                  int32_t* step, int32_t* out_tokens, int max_steps, void* ws,
                                  const Launch& L) {
  ArgmaxParams p = {};
  p.logits = logits;
  p.V = V;
  p.B = B;
  p.tok = tok;
  p.pos = pos;
  p.step = step;
  p.out = out_tokens;
  p.max_steps = max_steps;
  p.cand = (Cand*)ws;
  p.cnt = (int*)((unsigned char*)ws + (((size_t)B * kArgmaxBlocks * sizeof(Cand) + 255) & ~(size_t)255));
  p.err = L.err;
  const int blocks = std::min(kArgmaxBlocks, std::max(1, ceil_div(V, kArgmaxThreads * 4)));
  return launch_ex(argmax_advance_kernel, dim3(blocks, B), dim3(kArgmaxThreads), 0, L, p);
}

cudaError_t launch_embed(const void* embed, int H, int V, const int32_t* tok, int B, float* res,
                         const Launch& L) {
  const int threads = 256;
  const int blocks = std::max(1, std::min(8, ceil_div(H, threads * 8)));
  return launch_ex(embed_kernel, dim3(blocks, B), dim3(threads), 0, L, (const __nv_bfloat16*)embed, H,
                   V, tok, res, L.err);
}

cudaError_t launch_rmsnorm_rows(const float* x, const void* w, int B, int K, float eps, void* out_bf16,
                                const Launch& L) {
  if (K % 8 != 0) return cudaErrorInvalidValue;
  const int cpt = ceil_div(K / 8, 256);
  const __nv_bfloat16* wb = (const __nv_bfloat16*)w;
  __nv_bfloat16* ob = (__nv_bfloat16*)out_bf16;
  switch (cpt) {
    case 1: return launch_ex(rmsnorm_rows_kernel<1>, dim3(B), dim3(256), 0, L, x, wb, K, eps, ob);
    case 2: return launch_ex(rmsnorm_rows_kernel<2>, dim3(B), dim3(256), 0, L, x, wb, K, eps, ob);
    case 3: return launch_ex(rmsnorm_rows_kernel<3>, dim3(B), dim3(256), 0, L, x, wb, K, eps, ob);
    case 4: return launch_ex(rmsnorm_rows_kernel<4>, dim3(B), dim3(256), 0, L, x, wb, K, eps, ob);
    default: return cudaErrorInvalidValue;  // rows above 8192 are not a decode-step shape here
  }
}

cudaError_t launch_swiglu_rows(const float* gu, int B, int F, void* out_bf16, const Launch& L) {
  const int blocks = std::max(1, std::min(32, ceil_div(F, 256)));
  return launch_ex(swiglu_rows_kernel, dim3(blocks, B), dim3(256), 0, L, gu, F, (__nv_bfloat16*)out_bf16);
}

cudaError_t launch_paged_indices(const int32_t* pt, int B, int max_pages, int ps, int n_pages, int n_tokens,
                                 int32_t* idx, const Launch& L) {
  const long long n = (long long)B * n_tokens;
  if (n == 0) return cudaSuccess;
  return launch_ex(paged_indices_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, L, pt, B, max_pages, ps,
                   n_pages, n_tokens, idx, L.err);
}

}  // namespace qd
