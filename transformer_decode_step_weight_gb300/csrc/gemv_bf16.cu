// Weight-streaming BF16 GEMV for the decode step.
//
// "qwen3-8b-rtx4080-cutedsl" README, "Decode GEMV path" and "GPU Kernel Lab"
// README, "Fundamental kernels" (warp-reduced decode GEMV): at batch 1 every
// projection is y = W x with W streamed from HBM exactly once, so the kernel
// is a bandwidth kernel. "emit_qwen38_generate" rustdoc, "Where the speed comes
// from", item 1: projections that share an activation are concatenated rows of
// one matrix and run as one launch (QKV, gate+up).
//
// GB300 layout of the work:
//   * one CTA of up to 512 threads per SM (grid = #SMs); CTA i owns a
//     contiguous block of rows whose sizes differ by at most one, so every SM
//     streams the same number of bytes;
//   * inside a CTA, thread t of a row group owns fixed 16-byte column chunks
//     (8 bf16) of every row, so its slice of the activation vector lives in
//     registers for the whole kernel and each row is read as T x 16 B fully
//     coalesced segments; P row groups run side by side when a row needs fewer
//     than 512 threads;
//   * weights are loaded with 128-bit non-allocating, evict-first loads, U rows
//     x C chunks per thread in flight; the first batch is issued before the
//     programmatic-dependent-launch wait, so it overlaps the previous kernel;
//   * per row: warp-shuffle reduction, one partial per warp to shared memory,
//     then a fixed-order sum over warps (deterministic, no atomics).
// Fused prologues build the activation slice in registers: plain bf16/f32 x,
// the residual RMSNorm with the Qwen cast order (w * bf16(x * rsqrt(ms + eps)),
// "GPU Kernel Lab" README, "Fundamental kernels"), or SwiGLU (silu(g) * u) of
// the gate+up output. The residual-add epilogue does res[r] += y.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <algorithm>

namespace qd {
namespace {

constexpr int kThreads = 512;
constexpr int kSmemBudget = 96 * 1024;

struct GemvParams {
  const __nv_bfloat16* W;
  int R, K, batch;
  int rows_base, rows_extra;
  int T, P, phase_rows;
  int pro;
  const void* x;
  const __nv_bfloat16* norm_w;
  float eps;
  int epi;
  float* y;
};

QD_DEV float dot8(const uint4& w, const float* x) {
  float s = bf_lo(w.x) * x[0];
  s = fmaf(bf_hi(w.x), x[1], s);
  s = fmaf(bf_lo(w.y), x[2], s);
  s = fmaf(bf_hi(w.y), x[3], s);
  s = fmaf(bf_lo(w.z), x[4], s);
  s = fmaf(bf_hi(w.z), x[5], s);
  s = fmaf(bf_lo(w.w), x[6], s);
  s = fmaf(bf_hi(w.w), x[7], s);
  return s;
}

QD_DEV float silu(float g) { return g / (1.0f + expf(-g)); }

template <int C, int NB, int U>
__global__ void __launch_bounds__(kThreads, 1) gemv_bf16_kernel(const GemvParams p) {
  extern __shared__ float red[];
  __shared__ float s_ss[NB][kThreads / 32];

  const int tid = threadIdx.x;
  const int T = p.T, P = p.P, K = p.K;
  const int g = tid / T, t = tid - g * T;
  const int wpg = T >> 5, wig = t >> 5, lane = tid & 31;
  const int nrows = p.rows_base + ((int)blockIdx.x < p.rows_extra ? 1 : 0);
  const int r0 = (int)blockIdx.x * p.rows_base + min((int)blockIdx.x, p.rows_extra);
  const __nv_bfloat16* Wc = p.W + (size_t)r0 * K;

  int col[C];
  bool cv[C];
#pragma unroll
  for (int j = 0; j < C; ++j) {
    col[j] = (j * T + t) * 8;
    cv[j] = col[j] < K;
  }

  uint4 w[U][C];
  auto load_batch = [&](int ph0, int nph, int k0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int lr = g + P * (k0 + u);
      const bool ok = lr < nph;
      const __nv_bfloat16* rowp = Wc + (size_t)(ph0 + lr) * K;
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (ok && cv[j]) w[u][j] = ld_stream(rowp + col[j]);
        else w[u][j] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };

  const int nph_first = min(p.phase_rows, nrows);
  load_batch(0, nph_first, 0);  // weights do not depend on earlier kernels

  pdl_wait();
  pdl_launch_dependents();

  // ---- prologue: this thread's activation slice, x[b][j][0..7]
  float x[NB][C][8];
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int j = 0; j < C; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) x[b][j][e] = 0.f;

  if (p.pro == PRO_X_BF16) {
    const __nv_bfloat16* xb = (const __nv_bfloat16*)p.x;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b >= p.batch) break;
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (!cv[j]) continue;
        const uint4 v = *(const uint4*)(xb + (size_t)b * K + col[j]);
        x[b][j][0] = bf_lo(v.x); x[b][j][1] = bf_hi(v.x);
        x[b][j][2] = bf_lo(v.y); x[b][j][3] = bf_hi(v.y);
        x[b][j][4] = bf_lo(v.z); x[b][j][5] = bf_hi(v.z);
        x[b][j][6] = bf_lo(v.w); x[b][j][7] = bf_hi(v.w);
      }
    }
  } else if (p.pro == PRO_X_F32 || p.pro == PRO_RMSNORM) {
    const float* xf = (const float*)p.x;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b >= p.batch) break;
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (!cv[j]) continue;
        const float4 a = *(const float4*)(xf + (size_t)b * K + col[j]);
        const float4 c = *(const float4*)(xf + (size_t)b * K + col[j] + 4);
        x[b][j][0] = a.x; x[b][j][1] = a.y; x[b][j][2] = a.z; x[b][j][3] = a.w;
        x[b][j][4] = c.x; x[b][j][5] = c.y; x[b][j][6] = c.z; x[b][j][7] = c.w;
      }
    }
    if (p.pro == PRO_X_F32) {
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int j = 0; j < C; ++j)
#pragma unroll
          for (int e = 0; e < 8; ++e) x[b][j][e] = round_bf16(x[b][j][e]);
    } else {
      // RMSNorm over the K inputs of each sequence; row group 0 holds every column once.
      float ss[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float s = 0.f;
        if (g == 0) {
#pragma unroll
          for (int j = 0; j < C; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) s = fmaf(x[b][j][e], x[b][j][e], s);
        }
        s = warp_sum(s);
        if (lane == 0) s_ss[b][tid >> 5] = s;
      }
      __syncthreads();
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float s = 0.f;
        for (int i = 0; i < wpg; ++i) s += s_ss[b][i];  // group 0 = warps 0..wpg-1
        ss[b] = 1.0f / sqrtf(s / (float)K + p.eps);
      }
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (!cv[j]) continue;
        const uint4 wn = *(const uint4*)(p.norm_w + col[j]);
        float nw[8] = {bf_lo(wn.x), bf_hi(wn.x), bf_lo(wn.y), bf_hi(wn.y),
                       bf_lo(wn.z), bf_hi(wn.z), bf_lo(wn.w), bf_hi(wn.w)};
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int e = 0; e < 8; ++e)
            x[b][j][e] = (b < p.batch) ? round_bf16(nw[e] * round_bf16(x[b][j][e] * ss[b])) : 0.f;
      }
    }
  } else {  // PRO_SWIGLU: x = bf16(silu(g) * u), gate rows first, then up rows
    const float* gu = (const float*)p.x;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b >= p.batch) break;
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (!cv[j]) continue;
        const float* gp = gu + (size_t)b * 2 * K + col[j];
        const float4 g0 = *(const float4*)gp, g1 = *(const float4*)(gp + 4);
        const float4 u0 = *(const float4*)(gp + K), u1 = *(const float4*)(gp + K + 4);
        const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float uu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) x[b][j][e] = round_bf16(silu(gg[e]) * uu[e]);
      }
    }
  }

  // ---- main loop over phases of local rows
  for (int ph0 = 0; ph0 < nrows; ph0 += p.phase_rows) {
    const int nph = min(p.phase_rows, nrows - ph0);
    const int nk = (g < nph) ? (nph - g + P - 1) / P : 0;
    const int nbat = (nk + U - 1) / U;
    if (ph0 > 0) load_batch(ph0, nph, 0);
    for (int bi = 0; bi < nbat; ++bi) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int lr = g + P * (bi * U + u);
        if (lr < nph) {  // uniform across the warp
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < C; ++j) s += dot8(w[u][j], x[b][j]);
            s = warp_sum(s);
            if (lane == 0) red[(lr * NB + b) * wpg + wig] = s;
          }
        }
      }
      if (bi + 1 < nbat) load_batch(ph0, nph, (bi + 1) * U);
    }
    __syncthreads();
    for (int i = tid; i < nph * NB; i += blockDim.x) {
      const int lr = i / NB, b = i - lr * NB;
      if (b >= p.batch) continue;
      float s = 0.f;
      for (int k = 0; k < wpg; ++k) s += red[i * wpg + k];
      float* yp = p.y + (size_t)b * p.R + r0 + ph0 + lr;
      if (p.epi == EPI_RESID_ADD) *yp += s;
      else *yp = s;
    }
    __syncthreads();
  }
}

template <int C, int NB>
cudaError_t launch_cnb(const GemvParams& p, int grid, int threads, size_t smem, const Launch& L) {
  constexpr int U = (NB <= 2 ? 8 : 4) / C > 0 ? (NB <= 2 ? 8 : 4) / C : 1;
  auto k = gemv_bf16_kernel<C, NB, U>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(k, dim3(grid), dim3(threads), smem, L, p);
}

template <int C>
cudaError_t launch_c(const GemvParams& p, int nb, int grid, int threads, size_t smem, const Launch& L) {
  // batch x chunks per thread <= 8 keeps the activation slice in registers
  switch (nb) {
    case 1: return launch_cnb<C, 1>(p, grid, threads, smem, L);
    case 2: return launch_cnb<C, (C <= 4 ? 2 : 1)>(p, grid, threads, smem, L);
    case 4: return launch_cnb<C, (C <= 2 ? 4 : 1)>(p, grid, threads, smem, L);
    default: return launch_cnb<C, (C <= 1 ? 8 : 1)>(p, grid, threads, smem, L);
  }
}

int pick_c(int K) {
  const int chunks = K / 8;
  static const int opts[] = {1, 2, 3, 4, 6, 8};
  for (int c : opts)
    if (chunks <= c * kThreads) return c;
  return 0;
}

}  // namespace

bool gemv_bf16_supported(int K, int batch) {
  const int c = K > 0 && K % 8 == 0 ? pick_c(K) : 0;
  if (c == 0 || batch < 1 || batch > 8) return false;
  const int nb = batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : 8;
  return nb * c <= 8;
}

cudaError_t launch_gemv_bf16(const GemvBf16Args& a, const Launch& L) {
  const int C = pick_c(a.K);
  const int chunks = a.K / 8;
  const int T = std::min(kThreads, ((ceil_div(chunks, C) + 31) / 32) * 32);
  const int P = std::max(1, kThreads / T);
  const int threads = T * P;
  const int grid = std::max(1, std::min(a.R, dev_info().sm_count));
  const int nb = a.batch <= 1 ? 1 : a.batch <= 2 ? 2 : a.batch <= 4 ? 4 : 8;
  const int wpg = T / 32;
  const int rows_max = ceil_div(a.R, grid);
  const int per_row = nb * wpg * (int)sizeof(float);
  const int phase_rows = std::max(1, std::min(rows_max, kSmemBudget / per_row));

  GemvParams p;
  p.W = (const __nv_bfloat16*)a.W;
  p.R = a.R; p.K = a.K; p.batch = a.batch;
  p.rows_base = a.R / grid; p.rows_extra = a.R % grid;
  p.T = T; p.P = P; p.phase_rows = phase_rows;
  p.pro = a.pro; p.x = a.x; p.norm_w = (const __nv_bfloat16*)a.norm_w; p.eps = a.eps;
  p.epi = a.epi; p.y = a.y;
  const size_t smem = (size_t)phase_rows * per_row;
  switch (C) {
    case 1: return launch_c<1>(p, nb, grid, threads, smem, L);
    case 2: return launch_c<2>(p, nb, grid, threads, smem, L);
    case 3: return launch_c<3>(p, nb, grid, threads, smem, L);
    case 4: return launch_c<4>(p, nb, grid, threads, smem, L);
    case 6: return launch_c<6>(p, nb, grid, threads, smem, L);
    default: return launch_c<8>(p, nb, grid, threads, smem, L);
  }
}

}  // namespace qd
