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
#include <cstdlib>

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

QD_DEV float dot8(const uint4& w, const float* x) {  // two independent chains of four
  float a = bf_lo(w.x) * x[0], b = bf_hi(w.x) * x[1];
  a = fmaf(bf_lo(w.y), x[2], a);
  b = fmaf(bf_hi(w.y), x[3], b);
  a = fmaf(bf_lo(w.z), x[4], a);
  b = fmaf(bf_hi(w.z), x[5], b);
  a = fmaf(bf_lo(w.w), x[6], a);
  b = fmaf(bf_hi(w.w), x[7], b);
  return a + b;
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

// ---------------------------------------------------------------------------
// Batch-1 form on a TMA ring. One producer warp streams the CTA's contiguous
// weight rows into a shared-memory ring with cp.async.bulk (a few rows per
// stage, ~128 KB in flight per SM, issued before the programmatic-dependent
// wait because weights never depend on an earlier kernel); eight consumer
// warps own fixed 16-byte column chunks of every row (activation slice in
// registers), read the stage from shared memory, reduce each row with warp
// shuffles and a fixed-order sum over warps. The launcher pads the shared
// memory past half an SM so that exactly one GEMV CTA runs per SM (two on one
// SM under programmatic dependent launch made straggler CTAs); the next
// kernel's CTA takes the SM as soon as this one exits and starts its own ring
// before its dependency wait.
constexpr int kCons = 256;          // consumer threads
constexpr int kRingMax = 192 * 1024; // largest ring the launcher may choose
constexpr int kPhaseRows = 128;     // rows reduced per phase

struct RingParams {
  const __nv_bfloat16* W;
  int R, K;
  int ring_bytes;
  int rows_base, rows_extra;
  int T, P, rps, ns, stage_bytes;
  int pro;
  const void* x;
  const __nv_bfloat16* norm_w;
  float eps;
  int epi;
  float* y;
  int* err;
  int trig_late;
  L2Prefetch pf;
  int pair_F;                 // EPI_SWIGLU: F (rows of each half); the partition is over pairs
  __nv_bfloat16* y_bf16;      // EPI_SWIGLU output [F]
  int w_evict_first;          // weight copies marked evict-first in L2
};

QD_DEV void cons_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCons) : "memory"); }

template <int C, int RPS>
__global__ void __launch_bounds__(kCons + 32, 1) gemv_ring_kernel(const RingParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = (uint64_t*)(smem + p.ring_bytes);
  uint64_t* empty = full + 16;
  float* red = (float*)(empty + 16);            // [kPhaseRows][wpg]
  float* s_pair = red + kPhaseRows * (p.T / 32);  // EPI_SWIGLU: row sums [2 * npair]
  __shared__ float s_ss[kCons / 32];

  const int tid = threadIdx.x, lane = tid & 31;
  const int K = p.K, ns = p.ns;
  const bool pair = p.epi == EPI_SWIGLU;
  // r0: first row (first pair under EPI_SWIGLU); local rows [0, npair) are gate rows
  // r0.., local rows [npair, 2 npair) the up rows F + r0..
  const int nown = p.rows_base + ((int)blockIdx.x < p.rows_extra ? 1 : 0);
  const int npair = pair ? nown : 0;
  const int nrows = pair ? 2 * nown : nown;
  const int r0 = (int)blockIdx.x * p.rows_base + min((int)blockIdx.x, p.rows_extra);
  const int n_stages = (nrows + p.P * RPS - 1) / (p.P * RPS);
  const size_t row_bytes = (size_t)K * 2;

  if (tid == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCons / 32);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (!p.trig_late) pdl_launch_dependents();

  if (tid >= kCons) {  // ---- producer warp: weights only, so no dependency wait
    if (lane == 0) {
      const unsigned char* src = (const unsigned char*)(p.W + (size_t)r0 * K);
      // EPI_SWIGLU: local row lr >= npair is weight row F + r0 + (lr - npair)
      const unsigned char* src_up = pair ? (const unsigned char*)(p.W + ((size_t)p.pair_F + r0) * K) : src;
      const uint64_t pol = policy_evict_first();
      auto copy = [&](void* d, const void* g, uint32_t n, uint64_t* bar) {
        if (p.w_evict_first) bulk_g2s_hint(d, g, n, bar, pol);
        else bulk_g2s(d, g, n, bar);
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
          const int na = max(0, min(a + rows_i, npair) - a);   // gate rows in this stage
          if (na > 0) copy(dst, src + (size_t)a * row_bytes, (uint32_t)(na * row_bytes), &full[slot]);
          if (rows_i > na)
            copy(dst + (size_t)na * row_bytes, src_up + (size_t)(a + na - npair) * row_bytes,
                     (uint32_t)((rows_i - na) * row_bytes), &full[slot]);
        }
      }
    }
    __syncwarp();
    pdl_launch_dependents();  // every copy of this CTA is issued
    // This CTA's last ring refill is in flight: DRAM would go idle here while
    // the consumers drain, so fetch the head of the next GEMV's spans into L2.
    l2_prefetch_spans(p.pf, blockIdx.x, gridDim.x, lane);
    return;
  }

  // ---- consumers
  const int T = p.T, P = p.P;
  const int g = tid / T, t = tid - g * T;
  const int wpg = T >> 5, wig = t >> 5;
  int col[C];
  bool cv[C];
#pragma unroll
  for (int j = 0; j < C; ++j) {
    col[j] = (j * T + t) * 8;
    cv[j] = col[j] < K;
  }
  // the RMSNorm weights never come from an earlier kernel: load them before the wait
  uint4 wn[C];
#pragma unroll
  for (int j = 0; j < C; ++j)
    wn[j] = (p.pro == PRO_RMSNORM && cv[j]) ? *(const uint4*)(p.norm_w + col[j]) : make_uint4(0u, 0u, 0u, 0u);
  pdl_wait();

  float x[C][8];
#pragma unroll
  for (int j = 0; j < C; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) x[j][e] = 0.f;
  if (p.pro == PRO_X_BF16) {
    const __nv_bfloat16* xb = (const __nv_bfloat16*)p.x;
#pragma unroll
    for (int j = 0; j < C; ++j) {
      if (!cv[j]) continue;
      const uint4 v = *(const uint4*)(xb + col[j]);
      x[j][0] = bf_lo(v.x); x[j][1] = bf_hi(v.x); x[j][2] = bf_lo(v.y); x[j][3] = bf_hi(v.y);
      x[j][4] = bf_lo(v.z); x[j][5] = bf_hi(v.z); x[j][6] = bf_lo(v.w); x[j][7] = bf_hi(v.w);
    }
  } else if (p.pro == PRO_X_F32 || p.pro == PRO_RMSNORM) {
    const float* xf = (const float*)p.x;
#pragma unroll
    for (int j = 0; j < C; ++j) {
      if (!cv[j]) continue;
      const float4 a = *(const float4*)(xf + col[j]);
      const float4 c = *(const float4*)(xf + col[j] + 4);
      x[j][0] = a.x; x[j][1] = a.y; x[j][2] = a.z; x[j][3] = a.w;
      x[j][4] = c.x; x[j][5] = c.y; x[j][6] = c.z; x[j][7] = c.w;
    }
    if (p.pro == PRO_X_F32) {
#pragma unroll
      for (int j = 0; j < C; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) x[j][e] = round_bf16(x[j][e]);
    } else {
      float ss = 0.f;
      if (g == 0) {
#pragma unroll
        for (int j = 0; j < C; ++j)
#pragma unroll
          for (int e = 0; e < 8; ++e) ss = fmaf(x[j][e], x[j][e], ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) s_ss[tid >> 5] = ss;
      cons_sync();
      float tot = 0.f;
      for (int i = 0; i < wpg; ++i) tot += s_ss[i];
      const float inv = 1.0f / sqrtf(tot / (float)K + p.eps);
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (!cv[j]) continue;
        const float nw[8] = {bf_lo(wn[j].x), bf_hi(wn[j].x), bf_lo(wn[j].y), bf_hi(wn[j].y),
                             bf_lo(wn[j].z), bf_hi(wn[j].z), bf_lo(wn[j].w), bf_hi(wn[j].w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) x[j][e] = round_bf16(nw[e] * round_bf16(x[j][e] * inv));
      }
    }
  } else {  // PRO_SWIGLU
    const float* gu = (const float*)p.x;
#pragma unroll
    for (int j = 0; j < C; ++j) {
      if (!cv[j]) continue;
      const float* gp = gu + col[j];
      const float4 g0 = *(const float4*)gp, g1 = *(const float4*)(gp + 4);
      const float4 u0 = *(const float4*)(gp + K), u1 = *(const float4*)(gp + K + 4);
      const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const float uu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) x[j][e] = round_bf16(silu(gg[e]) * uu[e]);
    }
  }

  // stage = P groups x RPS rows; group g owns rows [g*RPS, g*RPS + RPS) of every stage
  const int stage_rows = P * RPS;
  int ph_base = 0;  // first local row of the current reduction phase
  for (int i = 0; i < n_stages; ++i) {
    const int slot = i % ns;
    if (!mbar_wait_bounded(&full[slot], (uint32_t)((i / ns) & 1), p.err)) {
      for (int k = 1; k < ns && i + k < n_stages; ++k)
        mbar_wait_bounded(&full[(i + k) % ns], (uint32_t)(((i + k) / ns) & 1), p.err);
      return;
    }
    if (i + 1 == n_stages) pdl_launch_dependents();
    const int row0 = i * stage_rows + g * RPS;          // local row of this group's first row
    const unsigned char* base = ring + (size_t)slot * p.stage_bytes + (size_t)g * RPS * row_bytes;
    const int nv = min(RPS, nrows - row0);              // valid rows of the group (may be <= 0)
    uint4 w[RPS][C];
#pragma unroll
    for (int r = 0; r < RPS; ++r)
#pragma unroll
      for (int j = 0; j < C; ++j)
        w[r][j] = (r < nv && cv[j]) ? *(const uint4*)(base + (size_t)r * row_bytes + (size_t)col[j] * 2)
                                    : make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);           // the stage is in registers now
    float v[RPS];
#pragma unroll
    for (int r = 0; r < RPS; ++r) {
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < C; ++j) a += dot8(w[r][j], x[j]);
      v[r] = a;
    }
    // transposed butterfly: after it, lane l holds the warp sum of row rsel(l)
    int rsel = 0;
#pragma unroll
    for (int L = 16, n = RPS; L >= 1; L >>= 1) {
      if (n > 1) {
        const int h = n / 2;
        const bool up = (lane & L) != 0;
#pragma unroll
        for (int k = 0; k < h; ++k) {
          const float send = up ? v[k] : v[k + h];
          const float keep = up ? v[k + h] : v[k];
          v[k] = keep + __shfl_xor_sync(0xffffffffu, send, L);
        }
        if (up) rsel += h;
        n = h;
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], L);
      }
    }
    constexpr int kLowMask = 32 / RPS - 1;              // lanes below the halving levels
    if ((lane & kLowMask) == 0 && rsel < nv)
      red[(row0 + rsel - ph_base) * wpg + wig] = v[0];
    const int done = min((i + 1) * stage_rows, nrows);
    if (done + stage_rows - ph_base > kPhaseRows || i + 1 == n_stages) {  // the next stage would not fit
      const int nph = done - ph_base;
      cons_sync();
      for (int r = tid; r < nph; r += kCons) {
        float acc = 0.f;
        for (int k = 0; k < wpg; ++k) acc += red[r * wpg + k];
        if (pair) {
          s_pair[ph_base + r] = acc;
        } else {
          float* yp = p.y + r0 + ph_base + r;
          if (p.epi == EPI_RESID_ADD) *yp += acc;
          else *yp = acc;
        }
      }
      cons_sync();
      ph_base = done;
    }
  }
  if (pair) {  // SwiGLU of the CTA's pairs (the last flush ended with a barrier)
    for (int j = tid; j < npair; j += kCons)
      p.y_bf16[r0 + j] = __float2bfloat16_rn(silu(s_pair[j]) * s_pair[npair + j]);
  }
}

template <int C>
cudaError_t launch_ring_c(const RingParams& p, int grid, size_t smem, const Launch& L) {
  constexpr int RPS = C == 1 ? 8 : C == 2 ? 4 : C <= 4 ? 2 : 1;
  auto k = gemv_ring_kernel<C, RPS>;
  static bool attr_set = false;
  if (!attr_set) {  // the largest size any launch of this kernel may ask for
    const int most = std::min(dev_info().max_smem_optin - 1024,
                              kRingMax + 32 * 8 + kPhaseRows * (kCons / 32) * 4 + 64 * 1024);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(k, dim3(grid), dim3(kCons + 32), smem, L, p);
}

}  // namespace

bool gemv_bf16_supported(int K, int batch) {
  const int c = K > 0 && K % 8 == 0 ? pick_c(K) : 0;
  if (c == 0 || batch < 1 || batch > 8) return false;
  const int nb = batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : 8;
  return nb * c <= 8;
}

static int ring_c(int K) {
  const int chunks = K / 8;
  static const int opts[] = {1, 2, 3, 4, 6};
  for (int c : opts)
    if (chunks <= c * kCons) return c;
  return 0;
}

// Ring geometry: a stage is P x RPS whole rows; the ring holds ~ring_kb KB of
// stages (default 128: measured 1.6 % faster on the Qwen3-8B step than 96, and
// 192 slower). The dynamic shared memory asked for is at least half of
// an SM's, so two GEMV CTAs never share an SM: with programmatic dependent
// launch the next GEMV's CTA would otherwise double up on the SMs that finish
// first and straggle (measured: 234 vs 295 tok/s on the Qwen3-8B step).
// QD_GEMV_RING_KB /
// QD_GEMV_SMEM_PAD_KB override the ring size / add padding (tuning);
// QD_GEMV_RING=0 selects the register-streaming kernel.
struct RingTuning {
  int enabled = 1, ring_kb = 128, pad_kb = 0, one_per_sm = 1;
  RingTuning() {
    if (const char* v = getenv("QD_GEMV_RING")) enabled = atoi(v) != 0;
    if (const char* v = getenv("QD_GEMV_ONE_PER_SM")) one_per_sm = atoi(v) != 0;
    if (const char* v = getenv("QD_GEMV_SMEM_PAD_KB")) pad_kb = std::max(0, std::min(64, atoi(v)));
    if (const char* v = getenv("QD_GEMV_RING_KB")) ring_kb = std::max(16, std::min(kRingMax / 1024, atoi(v)));
  }
};
static const RingTuning& ring_tuning() {
  static RingTuning t;
  return t;
}

L2Prefetch l2_plan_rows(const void* base, int R, size_t row_bytes, size_t head_bytes) {
  L2Prefetch pf = {};
  if (base == nullptr || R < 1 || row_bytes % 16 != 0 || ((uintptr_t)base & 15) != 0 || head_bytes < 16) return pf;
  const int grid = std::max(1, std::min(R, dev_info().sm_count));  // as every GEMV launcher cuts rows
  pf.base = base;
  pf.row_bytes = row_bytes;
  pf.rows_base = R / grid;
  pf.rows_extra = R % grid;
  pf.n_spans = grid;
  pf.head_bytes = head_bytes;
  return pf;
}

bool gemv_bf16_ring_ok(int K, int batch) {
  const int rc = (batch == 1 && ring_tuning().enabled && K % 8 == 0) ? ring_c(K) : 0;
  const int rps = rc == 1 ? 8 : rc == 2 ? 4 : rc <= 4 ? 2 : 1;
  return rc > 0 && (size_t)K * 2 * rps * 2 <= (size_t)kRingMax;
}

bool gemv_bf16_swiglu_ok(int K) {
  const int rc = gemv_bf16_ring_ok(K, 1) ? ring_c(K) : 0;
  return rc >= 1 && rc <= 4;  // RPS >= 2: a stage holds whole gate/up pairs
}

cudaError_t launch_gemv_bf16(const GemvBf16Args& a, const Launch& L) {
  const RingTuning& tu = ring_tuning();
  const int rc = (a.batch == 1 && tu.enabled) ? ring_c(a.K) : 0;
  const int ring_bytes = (a.ring_kb > 0 ? std::min(a.ring_kb, kRingMax / 1024) : tu.ring_kb) * 1024;
  const int rc_rps = rc == 1 ? 8 : rc == 2 ? 4 : rc <= 4 ? 2 : 1;
  if (rc > 0 && (size_t)a.K * 2 * rc_rps * 2 <= (size_t)kRingMax) {
    const int chunks = a.K / 8;
    RingParams p = {};
    p.W = (const __nv_bfloat16*)a.W;
    p.R = a.R; p.K = a.K;
    const bool pair = a.epi == EPI_SWIGLU;
    const int units = pair ? a.R / 2 : a.R;   // rows, or gate/up pairs
    const int grid = std::max(1, std::min(units, dev_info().sm_count));
    p.rows_base = units / grid; p.rows_extra = units % grid;
    p.pair_F = pair ? a.R / 2 : 0;
    p.y_bf16 = (__nv_bfloat16*)a.y_bf16;
    p.T = std::min(kCons, ((ceil_div(chunks, rc) + 31) / 32) * 32);
    p.P = std::max(1, kCons / p.T);
    const int row_bytes = a.K * 2;
    const int rps = rc == 1 ? 8 : rc == 2 ? 4 : rc <= 4 ? 2 : 1;     // must match launch_ring_c
    p.rps = rps;
    p.stage_bytes = ((p.P * rps * row_bytes + 127) / 128) * 128;
    p.ns = std::max(2, std::min(16, ring_bytes / p.stage_bytes));
    p.ring_bytes = p.ns * p.stage_bytes;
    p.pro = a.pro; p.x = a.x; p.norm_w = (const __nv_bfloat16*)a.norm_w; p.eps = a.eps;
    p.epi = a.epi; p.y = a.y; p.err = L.err; p.trig_late = L.trig_late;
    p.pf = a.pf;
    p.w_evict_first = a.w_evict_first;
    size_t smem = (size_t)p.ring_bytes + 32 * 8 + (size_t)kPhaseRows * (p.T / 32) * 4 + (size_t)tu.pad_kb * 1024;
    if (pair) smem += (size_t)2 * (p.rows_base + 1) * 4;
    if (smem > (size_t)dev_info().max_smem_optin - 1024) return cudaErrorInvalidValue;
    if (tu.one_per_sm) smem = std::max(smem, (size_t)dev_info().max_smem_optin / 2 + 1024);  // one GEMV CTA per SM
    switch (rc) {
      case 1: return launch_ring_c<1>(p, grid, smem, L);
      case 2: return launch_ring_c<2>(p, grid, smem, L);
      case 3: return launch_ring_c<3>(p, grid, smem, L);
      case 4: return launch_ring_c<4>(p, grid, smem, L);
      default: return launch_ring_c<6>(p, grid, smem, L);
    }
  }
  if (a.epi == EPI_SWIGLU) return cudaErrorInvalidValue;  // the ring form only
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

  GemvParams p = {};
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
