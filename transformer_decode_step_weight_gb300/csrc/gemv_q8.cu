// Q8_0 weight-streaming GEMV, both activation lanes, and the activation
// re-quantiser.
//
// "emit_qwen38_generate" rustdoc, "Where the speed comes from": at batch 1 a
// Q8_0 GEMV reads the whole weight matrix and one activation vector, so it is
// memory bound in either lane. ``deq`` selects the lane: activations kept in
// f32 and every weight dequantised (~3 float operations per weight), or the
// activation re-quantised per 32-block to int8 so the inner product is an
// exact int32 dp4a sum scaled by both block scales. Item 3 of the same section
// fuses the residual add, the next RMSNorm and the activation re-quantisation
// into one kernel: here they are the GEMV's prologue, computed per CTA.
//
// Layout: int8 values [R, K] and f16 scales [R, K/32] as two arrays. A thread
// owns C 16-weight half-blocks of every row of its CTA (one 16-byte value load
// and one 2-byte scale load each; the two halves of a block sit in adjacent
// lanes), so its activation slice — f32, or int8 plus scale — sits in
// registers. Dequantisation in the f32 lane builds each
// float from the byte with one byte-permute into the exponent pattern of 2^23
// and one exact subtraction (2^23 + u - (2^23 + 128) = q).
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <algorithm>
#include <cstdlib>

namespace qd {
namespace {

constexpr int kThreads = 512;
constexpr int kSmemBudget = 96 * 1024;

struct Q8Params {
  const int8_t* qs;
  const __half* d;
  int R, K;
  int rows_base, rows_extra;
  int T, P, phase_rows;
  int pro;
  const float* x;
  const int8_t* xq;
  const __half* xd;
  const __nv_bfloat16* norm_w;
  float eps;
  int epi;
  float* y;
  int32_t* dots;   // DUMP: the int32 block dots [R, K/32] this launch forms (i8 lane)
};

QD_DEV uint16_t ld_stream_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// 4 signed bytes -> 4 exact floats
QD_DEV void i8x4_to_f32(uint32_t w, float* f) {
  const uint32_t u = w ^ 0x80808080u;
  f[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)) - 8388736.0f;
  f[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541)) - 8388736.0f;
  f[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)) - 8388736.0f;
  f[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543)) - 8388736.0f;
}

QD_DEV float silu(float g) { return g / (1.0f + expf(-g)); }

// Exact int32 dot of a 16-weight half-block with the matching 16 int8 activation
// codes (four dp4a steps). Both GEMV forms use it; the two halves of a 32-block
// sit in adjacent lanes, so the block dot is this value plus the neighbour's.
QD_DEV int q8_half_dot(const uint32_t (&w)[4], const uint32_t (&x)[4]) {
  int acc = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) acc = __dp4a((int)w[k], (int)x[k], acc);
  return acc;
}

// Prologue that takes an already quantised activation (int8 + f16 scales).
constexpr int PRO_Q8_GIVEN = 16;

// DUMP: the i8 lane also stores each int32 block dot it forms (the test export
// of the bit-exact block dots runs the production kernel this way).
template <int C, int LANE, int U, bool DUMP>
__global__ void __launch_bounds__(kThreads, 1) gemv_q8_kernel(const Q8Params p) {
  extern __shared__ float red[];
  __shared__ float s_ss[kThreads / 32];
  const int tid = threadIdx.x;
  const int T = p.T, P = p.P, K = p.K, KB = p.K / 32, KC = p.K / 16;
  const int g = tid / T, t = tid - g * T;
  const int wpg = T >> 5, wig = t >> 5, lane = tid & 31;
  const int nrows = p.rows_base + ((int)blockIdx.x < p.rows_extra ? 1 : 0);
  const int r0 = (int)blockIdx.x * p.rows_base + min((int)blockIdx.x, p.rows_extra);

  // this thread owns 16-weight half-blocks ch[j] of every row (two threads per block)
  int ch[C];
  bool cv[C];
#pragma unroll
  for (int j = 0; j < C; ++j) {
    ch[j] = j * T + t;
    cv[j] = ch[j] < KC;
  }

  uint4 wq[U][C];
  uint16_t wd[U][C];
  auto load_batch = [&](int ph0, int nph, int k0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int lr = g + P * (k0 + u);
      const bool ok = lr < nph;
      const size_t r = (size_t)(r0 + ph0 + lr);
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (ok && cv[j]) {
          wq[u][j] = ld_stream(p.qs + r * K + (size_t)ch[j] * 16);
          wd[u][j] = ld_stream_u16(p.d + r * KB + (ch[j] >> 1));
        } else {
          wq[u][j] = make_uint4(0u, 0u, 0u, 0u);
          wd[u][j] = 0;
        }
      }
    }
  };

  load_batch(0, min(p.phase_rows, nrows), 0);
  pdl_wait();
  pdl_launch_dependents();

  // ---- activation half-blocks (f32), then the lane's form of them
  float xf[C][16];
  uint32_t xq[C][4];
  float xd[C];
#pragma unroll
  for (int j = 0; j < C; ++j) {
#pragma unroll
    for (int e = 0; e < 16; ++e) xf[j][e] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) xq[j][e] = 0u;
    xd[j] = 0.f;
  }
  if (p.pro == PRO_Q8_GIVEN) {
#pragma unroll
    for (int j = 0; j < C; ++j) {
      if (!cv[j]) continue;
      const uint4 a = *(const uint4*)(p.xq + (size_t)ch[j] * 16);
      xq[j][0] = a.x; xq[j][1] = a.y; xq[j][2] = a.z; xq[j][3] = a.w;
      xd[j] = __half2float(p.xd[ch[j] >> 1]);
    }
  } else {
    if (p.pro == PRO_SWIGLU) {
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (!cv[j]) continue;
        const float* gp = p.x + (size_t)ch[j] * 16;
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const float4 gg = *(const float4*)(gp + e), uu = *(const float4*)(gp + K + e);
          xf[j][e] = silu(gg.x) * uu.x;
          xf[j][e + 1] = silu(gg.y) * uu.y;
          xf[j][e + 2] = silu(gg.z) * uu.z;
          xf[j][e + 3] = silu(gg.w) * uu.w;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (!cv[j]) continue;
        const float* xp = p.x + (size_t)ch[j] * 16;
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const float4 a = *(const float4*)(xp + e);
          xf[j][e] = a.x; xf[j][e + 1] = a.y; xf[j][e + 2] = a.z; xf[j][e + 3] = a.w;
        }
      }
      if (p.pro == PRO_RMSNORM) {
        float s = 0.f;
        if (g == 0) {
#pragma unroll
          for (int j = 0; j < C; ++j)
#pragma unroll
            for (int e = 0; e < 16; ++e) s = fmaf(xf[j][e], xf[j][e], s);
        }
        s = warp_sum(s);
        if (lane == 0) s_ss[tid >> 5] = s;
        __syncthreads();
        float tot = 0.f;
        for (int i = 0; i < wpg; ++i) tot += s_ss[i];
        const float inv = 1.0f / sqrtf(tot / (float)K + p.eps);
#pragma unroll
        for (int j = 0; j < C; ++j) {
          if (!cv[j]) continue;
#pragma unroll
          for (int e = 0; e < 16; e += 8) {
            const uint4 wn = *(const uint4*)(p.norm_w + (size_t)ch[j] * 16 + e);
            const float nw[8] = {bf_lo(wn.x), bf_hi(wn.x), bf_lo(wn.y), bf_hi(wn.y),
                                 bf_lo(wn.z), bf_hi(wn.z), bf_lo(wn.w), bf_hi(wn.w)};
#pragma unroll
            for (int k = 0; k < 8; ++k) xf[j][e + k] = nw[k] * (xf[j][e + k] * inv);
          }
        }
      }
    }
    if (LANE == 1) {
      // re-quantise per 32-block: the two halves of a block sit in lanes t, t^1
#pragma unroll
      for (int j = 0; j < C; ++j) {
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(xf[j][e]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        const float d = amax / 127.0f;
        const float id = d != 0.0f ? 1.0f / d : 0.0f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t packed = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            int v = (int)roundf(xf[j][w * 4 + k] * id);
            v = max(-127, min(127, v));
            packed |= ((uint32_t)(v & 0xff)) << (8 * k);
          }
          xq[j][w] = packed;
        }
        xd[j] = __half2float(__float2half_rn(d));
      }
    }
  }

  for (int ph0 = 0; ph0 < nrows; ph0 += p.phase_rows) {
    const int nph = min(p.phase_rows, nrows - ph0);
    const int nk = (g < nph) ? (nph - g + P - 1) / P : 0;
    const int nbat = (nk + U - 1) / U;
    if (ph0 > 0) load_batch(ph0, nph, 0);
    for (int bi = 0; bi < nbat; ++bi) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int lr = g + P * (bi * U + u);
        if (lr < nph) {
          float s = 0.f;
#pragma unroll
          for (int j = 0; j < C; ++j) {
            const uint32_t wv[4] = {wq[u][j].x, wq[u][j].y, wq[u][j].z, wq[u][j].w};
            const float dw = __half2float(__ushort_as_half(wd[u][j]));
            if (LANE == 0) {
              float bs = 0.f;
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                float f[4];
                i8x4_to_f32(wv[w], f);
#pragma unroll
                for (int k = 0; k < 4; ++k) bs = fmaf(f[k], xf[j][w * 4 + k], bs);
              }
              s = fmaf(dw, bs, s);
            } else {
              const int acc = q8_half_dot(wv, xq[j]);
              if (DUMP) {
                const int other = __shfl_xor_sync(0xffffffffu, acc, 1);
                if ((t & 1) == 0 && cv[j]) p.dots[(size_t)(r0 + ph0 + lr) * KB + (ch[j] >> 1)] = acc + other;
              }
              s = fmaf((float)acc, dw * xd[j], s);
            }
          }
          s = warp_sum(s);
          if (lane == 0) red[lr * wpg + wig] = s;
        }
      }
      if (bi + 1 < nbat) load_batch(ph0, nph, (bi + 1) * U);
    }
    __syncthreads();
    for (int i = tid; i < nph; i += blockDim.x) {
      float s = 0.f;
      for (int k = 0; k < wpg; ++k) s += red[i * wpg + k];
      float* yp = p.y + r0 + ph0 + i;
      if (p.epi == EPI_RESID_ADD) *yp += s;
      else *yp = s;
    }
    __syncthreads();
  }
}

__global__ void quantize_q8_kernel(const float* x, int n, int8_t* xq, __half* xd) {
  const int blk = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (blk * 32 >= n) return;
  const float v = x[blk * 32 + lane];
  const float amax = warp_max(fabsf(v));
  const float d = amax / 127.0f;
  const float id = d != 0.0f ? 1.0f / d : 0.0f;
  int q = (int)roundf(v * id);
  q = max(-127, min(127, q));
  xq[blk * 32 + lane] = (int8_t)q;
  if (lane == 0) xd[blk] = __float2half_rn(d);
}

template <int C, int LANE, bool DUMP = false>
cudaError_t launch_cl(const Q8Params& p, int grid, int threads, size_t smem, const Launch& L) {
  constexpr int U = 8 / C;
  auto k = gemv_q8_kernel<C, LANE, U, DUMP>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(k, dim3(grid), dim3(threads), smem, L, p);
}

int pick_c(int K) {
  const int chunks = K / 16;
  static const int opts[] = {1, 2, 4};
  for (int c : opts)
    if (chunks <= c * kThreads) return c;
  return 0;
}

// ---------------------------------------------------------------------------
// Batch-1 Q8_0 GEMV on a TMA ring (same structure as the BF16 ring kernel): a
// producer warp streams each stage's rows of int8 values and their fp16 scales
// with two cp.async.bulk copies; eight consumer warps own 16-weight half-blocks
// of every row with the activation slice (f32, or int8 + scale) in registers.
constexpr int kConsQ = 256;
constexpr int kRingQMax = 200 * 1024;   // largest ring a launch may take
constexpr int kPhaseQ = 128;
// Ring bytes per lane (QD_Q8_RING_KB overrides both, read once). The dp4a lane is
// latency-bound, so more bytes in flight help it: at 24576 x 4096 it streamed 4.46 /
// 4.71 / 4.71 / 4.65 TB/s with 96 / 128 / 160 / 192 KB (Qwen3-8B Q8_0 step 485 -> 510
// tok/s at 160); the f32 lane is issue-bound and keeps 96 KB (398 vs 391 tok/s).
int ring_q_bytes(int act) {
  static const int forced = [] {
    const char* e = getenv("QD_Q8_RING_KB");
    return e ? std::max(64, std::min(200, atoi(e))) * 1024 : 0;
  }();
  if (forced) return forced;
  return (act == 1 ? 160 : 96) * 1024;
}

struct RingQ8Params {
  const int8_t* qs;
  const __half* d;
  int R, K;
  int rows_base, rows_extra;
  int T, P, ns, stage_bytes, ring_bytes;
  int pro;
  const float* x;
  const int8_t* xq;
  const __half* xd;
  const __nv_bfloat16* norm_w;
  float eps;
  int epi;
  float* y;
  int* err;
  int trig_late;
  int pair_F;            // EPI_SWIGLU: rows of each half; units are (gate j, up F + j) pairs
  int w_evict_first;
  int* claim;            // null: static split; else [claim, done] counters
  int static_per_cta;
  int32_t* dots;         // DUMP: the int32 block dots [R, K/32] this launch forms (i8 lane)
};

QD_DEV void cons_sync_q() { asm volatile("bar.sync 1, %0;" ::"n"(kConsQ) : "memory"); }
QD_DEV void mbar_arrive_q(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int C, int LANE, int RPS, bool DUMP>
__global__ void __launch_bounds__(kConsQ + 32, 1) gemv_q8_ring_kernel(const RingQ8Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = (uint64_t*)(smem + p.ring_bytes);
  uint64_t* empty = full + 16;
  int* st_u0 = (int*)(empty + 16);              // [16] first unit of each stage's chunk
  int* st_n = st_u0 + 16;                       // [16] units in it (0: no more work)
  float* red = (float*)(st_n + 16);             // [kPhaseQ][wpg]
  float* rsum = red + kPhaseQ * (p.T / 32);     // [kPhaseQ] EPI_SWIGLU: gate/up sums by pair slot
  int* rid = (int*)(rsum + kPhaseQ);            // [kPhaseQ] destination of each phase row
  int* pid = rid + kPhaseQ;                     // [kPhaseQ / 2] EPI_SWIGLU: pair of each pair slot
  __shared__ float s_ss[kConsQ / 32];

  const int tid = threadIdx.x, lane = tid & 31;
  const int K = p.K, KB = K / 32, KC = K / 16, ns = p.ns;
  const bool pair = p.epi == EPI_SWIGLU;
  // units: rows, or under EPI_SWIGLU (gate row j, up row F + j) pairs; static share
  // first, then (with a claim counter) stages of the pool [pool0, units)
  const int upr = pair ? 2 : 1;
  const int srows = p.P * RPS;
  const int cu = srows / upr;
  const int units = pair ? p.pair_F : p.R;
  int u_s, n_s;
  if (p.claim) {
    u_s = (int)blockIdx.x * p.static_per_cta;
    n_s = p.static_per_cta;
  } else {
    n_s = p.rows_base + ((int)blockIdx.x < p.rows_extra ? 1 : 0);
    u_s = (int)blockIdx.x * p.rows_base + min((int)blockIdx.x, p.rows_extra);
  }
  const int pool0 = p.claim ? p.static_per_cta * (int)gridDim.x : units;
  const size_t qrow = (size_t)K, drow = (size_t)KB * 2;   // bytes per row of values / scales
  const size_t dbase = (size_t)srows * qrow;               // scales follow the values in a stage

  if (tid == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsQ / 32);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (!p.trig_late) pdl_launch_dependents();

  if (tid >= kConsQ) {  // ---- producer warp: weights only
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      auto copy = [&](void* d, const void* g, uint32_t n, uint64_t* bar) {
        if (p.w_evict_first) bulk_g2s_hint(d, g, n, bar, pol);
        else bulk_g2s(d, g, n, bar);
      };
      const unsigned char* Q = (const unsigned char*)p.qs;
      const unsigned char* D = (const unsigned char*)p.d;
      int u = u_s;
      const int u_end = u_s + n_s;
      int next = p.claim ? pool0 + atomicAdd(p.claim, cu) : units;  // claimed one chunk ahead
      bool ok = true;
      int i = 0;
      for (;; ++i) {
        int c0, cn;
        if (u < u_end) {
          c0 = u;
          cn = min(cu, u_end - u);
          u += cn;
        } else {
          if (next >= units) break;
          c0 = next;
          cn = min(cu, units - c0);
          next = pool0 + atomicAdd(p.claim, cu);
        }
        const int slot = i % ns;
        if (i >= ns && !mbar_wait_bounded(&empty[slot], (uint32_t)(((i / ns) - 1) & 1), p.err)) {
          ok = false;
          break;
        }
        st_u0[slot] = c0;
        st_n[slot] = cn;
        unsigned char* st = ring + (size_t)slot * p.stage_bytes;
        mbar_arrive_expect_tx(&full[slot], (uint32_t)((size_t)cn * upr * (qrow + drow)));
        copy(st, Q + (size_t)c0 * qrow, (uint32_t)(cn * qrow), &full[slot]);
        copy(st + dbase, D + (size_t)c0 * drow, (uint32_t)(cn * drow), &full[slot]);
        if (pair) {
          const size_t up = (size_t)p.pair_F + c0;
          copy(st + (size_t)cn * qrow, Q + up * qrow, (uint32_t)(cn * qrow), &full[slot]);
          copy(st + dbase + (size_t)cn * drow, D + up * drow, (uint32_t)(cn * drow), &full[slot]);
        }
      }
      // Every copy of this CTA is issued: let the next kernel launch now (its weight
      // stream starts before its dependency wait). The end marker below may have to
      // wait for a free stage, and the trigger must not wait with it.
      pdl_launch_dependents();
      if (ok) {  // end marker: a stage of no units
        const int slot = i % ns;
        if (i < ns || mbar_wait_bounded(&empty[slot], (uint32_t)(((i / ns) - 1) & 1), p.err)) {
          st_n[slot] = 0;
          mbar_arrive_q(&full[slot]);
        }
      }
      if (p.claim) {  // the last producer to stop claiming resets the counters
        __threadfence();
        if (atomicAdd(p.claim + 1, 1) == (int)gridDim.x - 1) {
          atomicExch(p.claim, 0);
          atomicExch(p.claim + 1, 0);
        }
      }
    }
    __syncwarp();
    pdl_launch_dependents();
    return;
  }

  // ---- consumers: thread t of group g owns half-blocks ch[j] = j*T + t of every row
  const int T = p.T;
  const int g = tid / T, t = tid - g * T;
  const int wpg = T >> 5, wig = t >> 5;
  int ch[C];
  bool cv[C];
#pragma unroll
  for (int j = 0; j < C; ++j) {
    ch[j] = j * T + t;
    cv[j] = ch[j] < KC;
  }
  // the RMSNorm weights never come from an earlier kernel: load them before the wait
  uint4 wn[C][2];
#pragma unroll
  for (int j = 0; j < C; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h)
      wn[j][h] = (p.pro == PRO_RMSNORM && cv[j]) ? *(const uint4*)(p.norm_w + (size_t)ch[j] * 16 + h * 8)
                                                 : make_uint4(0u, 0u, 0u, 0u);
  pdl_wait();

  float xf[C][16];
  uint32_t xq[C][4];
  float xd[C];
#pragma unroll
  for (int j = 0; j < C; ++j) {
#pragma unroll
    for (int e = 0; e < 16; ++e) xf[j][e] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) xq[j][e] = 0u;
    xd[j] = 0.f;
  }
  if (p.pro == PRO_Q8_GIVEN) {
#pragma unroll
    for (int j = 0; j < C; ++j) {
      if (!cv[j]) continue;
      const uint4 a = *(const uint4*)(p.xq + (size_t)ch[j] * 16);
      xq[j][0] = a.x; xq[j][1] = a.y; xq[j][2] = a.z; xq[j][3] = a.w;
      xd[j] = __half2float(p.xd[ch[j] >> 1]);
    }
  } else {
    if (p.pro == PRO_SWIGLU) {
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (!cv[j]) continue;
        const float* gp = p.x + (size_t)ch[j] * 16;
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const float4 gg = *(const float4*)(gp + e), uu = *(const float4*)(gp + K + e);
          xf[j][e] = silu(gg.x) * uu.x;
          xf[j][e + 1] = silu(gg.y) * uu.y;
          xf[j][e + 2] = silu(gg.z) * uu.z;
          xf[j][e + 3] = silu(gg.w) * uu.w;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (!cv[j]) continue;
        const float* xp = p.x + (size_t)ch[j] * 16;
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const float4 a = *(const float4*)(xp + e);
          xf[j][e] = a.x; xf[j][e + 1] = a.y; xf[j][e + 2] = a.z; xf[j][e + 3] = a.w;
        }
      }
      if (p.pro == PRO_RMSNORM) {
        float ss = 0.f;
        if (g == 0) {
#pragma unroll
          for (int j = 0; j < C; ++j)
#pragma unroll
            for (int e = 0; e < 16; ++e) ss = fmaf(xf[j][e], xf[j][e], ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) s_ss[tid >> 5] = ss;
        cons_sync_q();
        float tot = 0.f;
        for (int i = 0; i < wpg; ++i) tot += s_ss[i];
        const float inv = 1.0f / sqrtf(tot / (float)K + p.eps);
#pragma unroll
        for (int j = 0; j < C; ++j) {
          if (!cv[j]) continue;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 w = wn[j][h];
            const float nw[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y),
                                 bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
#pragma unroll
            for (int k = 0; k < 8; ++k) xf[j][h * 8 + k] = nw[k] * (xf[j][h * 8 + k] * inv);
          }
        }
      }
    }
    if (LANE == 1) {  // re-quantise per 32-block; its halves sit in lanes t, t^1
#pragma unroll
      for (int j = 0; j < C; ++j) {
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(xf[j][e]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        const float dd = amax / 127.0f;
        const float id = dd != 0.0f ? 1.0f / dd : 0.0f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t packed = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            int v = (int)roundf(xf[j][w * 4 + k] * id);
            v = max(-127, min(127, v));
            packed |= ((uint32_t)(v & 0xff)) << (8 * k);
          }
          xq[j][w] = packed;
        }
        xd[j] = __half2float(__float2half_rn(dd));
      }
    }
  }

  int ph_n = 0, pp_n = 0;  // rows and (EPI_SWIGLU) pairs of the current phase
  auto flush = [&]() {
    cons_sync_q();
    for (int r = tid; r < ph_n; r += kConsQ) {
      float acc = 0.f;
      for (int k = 0; k < wpg; ++k) acc += red[r * wpg + k];
      if (pair) {
        rsum[rid[r]] = acc;
      } else {
        float* yp = p.y + rid[r];
        if (p.epi == EPI_RESID_ADD) *yp += acc;
        else *yp = acc;
      }
    }
    cons_sync_q();
    if (pair) {  // SwiGLU of the phase's pairs (f32, the value the down projection quantises)
      for (int q = tid; q < pp_n; q += kConsQ) p.y[pid[q]] = silu(rsum[2 * q]) * rsum[2 * q + 1];
      cons_sync_q();
    }
    ph_n = 0;
    pp_n = 0;
  };
  for (int i = 0;; ++i) {
    const int slot = i % ns;
    if (!mbar_wait_bounded(&full[slot], (uint32_t)((i / ns) & 1), p.err)) {
      for (int k = 1; k < ns; ++k)  // let copies still in flight land before the CTA leaves
        mbar_wait_bounded(&full[(i + k) % ns], (uint32_t)(((i + k) / ns) & 1), p.err);
      return;
    }
    const int c0 = st_u0[slot], cn = st_n[slot];
    if (cn == 0) break;
    const int svalid = cn * upr;                        // valid rows of the stage
    const int row0 = g * RPS;                           // this group's first row of the stage
    const unsigned char* st = ring + (size_t)slot * p.stage_bytes;
    const int nv = min(RPS, svalid - row0);
    uint4 wv[RPS][C];
    float dw[RPS][C];
#pragma unroll
    for (int r = 0; r < RPS; ++r)
#pragma unroll
      for (int j = 0; j < C; ++j) {
        const bool ok = r < nv && cv[j];
        const size_t lr = (size_t)(row0 + r);
        wv[r][j] = ok ? *(const uint4*)(st + lr * qrow + (size_t)ch[j] * 16) : make_uint4(0u, 0u, 0u, 0u);
        dw[r][j] = ok ? __half2float(*(const __half*)(st + dbase + lr * drow + (size_t)(ch[j] >> 1) * 2)) : 0.f;
      }
    __syncwarp();
    if (lane == 0) mbar_arrive_q(&empty[slot]);
    float v[RPS];
#pragma unroll
    for (int r = 0; r < RPS; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < C; ++j) {
        const uint32_t w4[4] = {wv[r][j].x, wv[r][j].y, wv[r][j].z, wv[r][j].w};
        if (LANE == 0) {
          float bs = 0.f, bs2 = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            float f[4];
            i8x4_to_f32(w4[w], f);
            bs = fmaf(f[0], xf[j][w * 4], bs);
            bs2 = fmaf(f[1], xf[j][w * 4 + 1], bs2);
            bs = fmaf(f[2], xf[j][w * 4 + 2], bs);
            bs2 = fmaf(f[3], xf[j][w * 4 + 3], bs2);
          }
          acc = fmaf(dw[r][j], bs + bs2, acc);
        } else {
          const int dot = q8_half_dot(w4, xq[j]);
          if (DUMP) {  // rows are units here (EPI_STORE): stage unit c0 + local row
            const int other = __shfl_xor_sync(0xffffffffu, dot, 1);
            if ((t & 1) == 0 && r < nv && cv[j]) p.dots[(size_t)(c0 + row0 + r) * KB + (ch[j] >> 1)] = dot + other;
          }
          acc = fmaf((float)dot, dw[r][j] * xd[j], acc);
        }
      }
      v[r] = acc;
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
          const float keep = up ? v[k + h] : v[k];
          v[k] = keep + __shfl_xor_sync(0xffffffffu, send, L);
        }
        if (up) rsel += h;
        n = h;
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], L);
      }
    }
    constexpr int kLowMask = 32 / RPS - 1;
    if ((lane & kLowMask) == 0 && rsel < nv) red[(ph_n + row0 + rsel) * wpg + wig] = v[0];
    if (tid < svalid) {  // destinations of the stage's rows
      if (pair) {
        const bool up_row = tid >= cn;
        const int q = up_row ? tid - cn : tid;
        rid[ph_n + tid] = 2 * (pp_n + q) + (up_row ? 1 : 0);
        if (!up_row) pid[pp_n + q] = c0 + q;
      } else {
        rid[ph_n + tid] = c0 + tid;
      }
    }
    ph_n += svalid;
    pp_n += pair ? cn : 0;
    if (ph_n + srows > kPhaseQ) flush();  // the next stage might not fit
  }
  if (p.trig_late) pdl_launch_dependents();
  flush();
}

template <int C, int LANE, bool DUMP = false>
cudaError_t launch_ring_q(const RingQ8Params& p, int grid, size_t smem, const Launch& L) {
  constexpr int RPS = C == 1 ? 8 : C == 2 ? 4 : 2;
  auto k = gemv_q8_ring_kernel<C, LANE, RPS, DUMP>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         dev_info().max_smem_optin - 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(k, dim3(grid), dim3(kConsQ + 32), smem, L, p);
}

// percent of a step GEMV's units claimed from the shared pool (QD_GEMV_DYN_PCT, as the BF16 ring)
int q8_dyn_pct() {
  static const int v = [] {
    const char* e = getenv("QD_GEMV_DYN_PCT");
    return e ? std::max(0, std::min(100, atoi(e))) : 15;
  }();
  return v;
}

int ring_q_c(int K) {
  const int chunks = K / 16;
  static const int opts[] = {1, 2, 3, 4};
  for (int c : opts)
    if (chunks <= c * kConsQ) return c;
  return 0;
}

}  // namespace

bool gemv_q8_supported(int K) { return K > 0 && K % 32 == 0 && pick_c(K) > 0; }

bool gemv_q8_swiglu_ok(int K) {
  const int rc = K % 256 == 0 ? ring_q_c(K) : 0;
  return rc >= 1;  // every ring form has RPS >= 2, so a stage holds whole gate/up pairs
}

cudaError_t launch_gemv_q8(const GemvQ8Args& a, const Launch& L) {
  if (a.dots && (a.act != 1 || a.epi != EPI_STORE)) return cudaErrorInvalidValue;  // i8 lane, plain rows
  const bool aligned = (((uintptr_t)a.qs | (uintptr_t)a.d) & 15) == 0;
  const int rc = (a.K % 256 == 0 && aligned) ? ring_q_c(a.K) : 0;
  if (rc > 0) {
    const int rps = rc == 1 ? 8 : rc == 2 ? 4 : 2;   // must match launch_ring_q
    RingQ8Params p = {};
    p.qs = a.qs; p.d = (const __half*)a.d; p.R = a.R; p.K = a.K;
    const bool pair = a.epi == EPI_SWIGLU;
    const int units = pair ? a.R / 2 : a.R;   // rows, or gate/up pairs
    const int grid = std::max(1, std::min(units, dev_info().sm_count));
    p.rows_base = units / grid; p.rows_extra = units % grid;
    p.pair_F = pair ? a.R / 2 : 0;
    if (pair && (std::max(1, kConsQ / std::min(kConsQ, ((ceil_div(a.K / 16, rc) + 31) / 32) * 32)) * rps) % 2 != 0)
      return cudaErrorInvalidValue;  // a stage holds whole pairs
    p.w_evict_first = a.w_evict_first;
    const int cu_q = (std::max(1, kConsQ / std::min(kConsQ, ((ceil_div(a.K / 16, rc) + 31) / 32) * 32)) * rps) /
                     (pair ? 2 : 1);
    if (a.claim && q8_dyn_pct() > 0 && units / grid >= 8 * cu_q) {  // as the BF16 ring: small chunks only
      p.claim = a.claim;
      p.static_per_cta = (int)(((long long)units * (100 - q8_dyn_pct())) / (100LL * grid));
    }
    p.T = std::min(kConsQ, ((ceil_div(a.K / 16, rc) + 31) / 32) * 32);
    p.P = std::max(1, kConsQ / p.T);
    const size_t row_bytes = (size_t)a.K + (size_t)a.K / 16;
    p.stage_bytes = (int)((((size_t)p.P * rps * row_bytes) + 127) / 128 * 128);
    p.ns = std::max(2, std::min(16, ring_q_bytes(a.act) / p.stage_bytes));
    p.ring_bytes = p.ns * p.stage_bytes;
    p.pro = a.pro; p.x = (const float*)a.x; p.xq = a.xq; p.xd = (const __half*)a.xd;
    if (a.act == 1 && a.xq != nullptr) p.pro = PRO_Q8_GIVEN;
    p.norm_w = (const __nv_bfloat16*)a.norm_w; p.eps = a.eps; p.epi = a.epi; p.y = a.y;
    p.err = L.err; p.trig_late = L.trig_late;
    size_t smem = (size_t)p.ring_bytes + 32 * 8 + 32 * 4 + (size_t)kPhaseQ * (p.T / 32) * 4 +
                  (size_t)kPhaseQ * 4 * 2 + (size_t)kPhaseQ / 2 * 4;
    smem = std::max(smem, (size_t)dev_info().max_smem_optin / 2 + 1024);  // one GEMV CTA per SM
    p.dots = a.dots;
    if ((size_t)p.ns * p.stage_bytes <= (size_t)kRingQMax) {
      if (a.dots) {
        switch (rc) {
          case 1: return launch_ring_q<1, 1, true>(p, grid, smem, L);
          case 2: return launch_ring_q<2, 1, true>(p, grid, smem, L);
          case 3: return launch_ring_q<3, 1, true>(p, grid, smem, L);
          default: return launch_ring_q<4, 1, true>(p, grid, smem, L);
        }
      }
      switch (rc) {
        case 1: return a.act == 1 ? launch_ring_q<1, 1>(p, grid, smem, L) : launch_ring_q<1, 0>(p, grid, smem, L);
        case 2: return a.act == 1 ? launch_ring_q<2, 1>(p, grid, smem, L) : launch_ring_q<2, 0>(p, grid, smem, L);
        case 3: return a.act == 1 ? launch_ring_q<3, 1>(p, grid, smem, L) : launch_ring_q<3, 0>(p, grid, smem, L);
        default: return a.act == 1 ? launch_ring_q<4, 1>(p, grid, smem, L) : launch_ring_q<4, 0>(p, grid, smem, L);
      }
    }
  }
  if (a.epi == EPI_SWIGLU) return cudaErrorInvalidValue;  // the ring form only
  const int C = pick_c(a.K);
  const int KC = a.K / 16;
  const int T = std::min(kThreads, ((ceil_div(KC, C) + 31) / 32) * 32);
  const int P = std::max(1, kThreads / T);
  const int threads = T * P;
  const int grid = std::max(1, std::min(a.R, dev_info().sm_count));
  const int wpg = T / 32;
  const int rows_max = ceil_div(a.R, grid);
  const int phase_rows = std::max(1, std::min(rows_max, kSmemBudget / (wpg * 4)));
  Q8Params p = {};
  p.qs = a.qs;
  p.d = (const __half*)a.d;
  p.R = a.R; p.K = a.K;
  p.rows_base = a.R / grid; p.rows_extra = a.R % grid;
  p.T = T; p.P = P; p.phase_rows = phase_rows;
  p.pro = a.pro; p.x = (const float*)a.x; p.norm_w = (const __nv_bfloat16*)a.norm_w; p.eps = a.eps;
  p.xq = a.xq; p.xd = (const __half*)a.xd;
  if (a.act == 1 && a.xq != nullptr) p.pro = PRO_Q8_GIVEN;
  p.epi = a.epi; p.y = a.y;
  p.dots = a.dots;
  const size_t smem = (size_t)phase_rows * wpg * 4;
  if (a.dots) {
    switch (C) {
      case 1: return launch_cl<1, 1, true>(p, grid, threads, smem, L);
      case 2: return launch_cl<2, 1, true>(p, grid, threads, smem, L);
      default: return launch_cl<4, 1, true>(p, grid, threads, smem, L);
    }
  }
  switch (C) {
    case 1: return a.act == 1 ? launch_cl<1, 1>(p, grid, threads, smem, L) : launch_cl<1, 0>(p, grid, threads, smem, L);
    case 2: return a.act == 1 ? launch_cl<2, 1>(p, grid, threads, smem, L) : launch_cl<2, 0>(p, grid, threads, smem, L);
    default: return a.act == 1 ? launch_cl<4, 1>(p, grid, threads, smem, L) : launch_cl<4, 0>(p, grid, threads, smem, L);
  }
}

cudaError_t launch_quantize_q8(const float* x, int n, int8_t* xq, void* xd, const Launch& L) {
  const int threads = 256;
  const int blocks = ceil_div((long long)n, threads);
  if (blocks == 0) return cudaSuccess;
  return launch_ex(quantize_q8_kernel, dim3(blocks), dim3(threads), 0, L, x, n, xq, (__half*)xd);
}

}  // namespace qd
