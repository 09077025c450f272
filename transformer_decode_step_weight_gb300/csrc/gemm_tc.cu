// Batched decode projections on the 5th-generation tensor cores (tcgen05).
//
// With B concurrent sequences the decode-step projections are the dense
// contraction Y[B, R] = X[B, K] . W[R, K]^T ("qwen3-8b-rtx4080-cutedsl" README,
// "Baseline tiled GEMM" / "Speculative decoding": a batch of tokens reuses the
// weight bytes already streamed). At B = 64 each weight element feeds 64 MACs,
// more than the CUDA cores can issue at HBM rate, so the contraction runs on
// tcgen05 with the weights as the M operand:
//   * one CTA per 128-row tile of W; D[128 rows x 64 tokens] accumulates in
//     TMEM (64 columns of f32), K advances in 64-element (128-byte) chunks;
//   * a producer thread streams W tiles [128 x 64] and X tiles [64 x 64] with
//     2D TMA (cp.async.bulk.tensor, 128-byte swizzle) through a 6-stage ring on
//     mbarriers; W loads are issued before the programmatic-dependent wait;
//   * one thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> f32, M=128,
//     N=64, K=16 per instruction) from shared-memory descriptors and commits
//     each stage back to the producer; a final commit releases the epilogue;
//   * the four warps read their 32 TMEM lanes each (tcgen05.ld 32x32b.x64) and
//     store y or add it to the residual stream.
// Q8_0 weights (int8 values, an fp16 scale per 32 of a row; "emit_qwen38_generate"
// rustdoc, "Where the speed comes from") take the same MMA and epilogue in a
// 384-thread form: warp 0 streams the int8 tiles [128 x 64 B] and their scale boxes
// with TMA, warp 2 the X tiles, and four groups of two converter warps widen each
// weight to bf16(f32(d) * q) (exact product, one round to nearest even) into the
// swizzled A tile the MMA reads, each group a different K step. The tensor cores'
// int8 rate on this part is far below their bf16 rate, so the int8 values are not
// fed to them directly.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace qd {
namespace {

constexpr int kBM = 128;        // weight rows per tile (MMA M)
constexpr int kBN = 64;         // tokens (MMA N, TMEM columns)
constexpr int kBK = 64;         // K elements per stage (128 bytes of bf16)
// bf16 ring depth: 6 stages (one CTA per SM) when the CTAs fit in one wave, else 3
// (~74 KB, two or three CTAs per SM, so a grid of up to twice the SM count still
// runs in one wave). QD_GEMM_STAGES = 3 or 6 forces one. The Q8_0 form's rings
// are set below (kQSt, kBSt, kASt).
constexpr int kTileA = kBM * kBK * 2;    // 16 KB
constexpr int kTileQ = kBM * kBK;        // 8 KB: int8 values of a Q8_0 tile
constexpr int kTileS = kBM * 16;         // 2 KB: 8 fp16 scales (256 columns) per row
constexpr int kThreadsTc = 128;
constexpr int kConvWarps = 8;            // Q8_0: warps 4..11 widen int8 -> bf16
constexpr int kThreadsQ8 = kThreadsTc + 32 * kConvWarps;
constexpr int kMaxSplits = 4;   // K splits of one tile (partials summed in registers)

struct TcParams {
  int R, K, B;
  int epi;        // EPI_STORE / EPI_RESID_ADD
  float* y;       // [B, R]
  int* err;
  int splits;     // K splits (grid y); > 1: partials through part / cnt
  float* part;    // [tiles][splits][kBN][kBM] f32 partial tiles
  int* cnt;       // [tiles] tickets, zero between launches
  int zfast;      // many rows: grid x = token tiles, y = weight tiles (the token tiles of a
                  // weight tile run together and share it through L2)
};

// --- tcgen05 / TMA wrappers -------------------------------------------------

QD_DEV void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
QD_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
QD_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
QD_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand tile of 128-byte rows with
// the 128-byte swizzle, 8-row groups 1024 bytes apart.
QD_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);          // start address
  d |= (uint64_t)1 << 16;                          // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                          // descriptor version
  d |= (uint64_t)2 << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor: D f32, A and B bf16, both K-major, M = 128, N = bn.
__host__ __device__ constexpr uint32_t idesc_for(int bn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

template <int BN>
QD_DEV void mma_bf16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t accumulate) {
  constexpr uint32_t kIdesc = idesc_for(BN);
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
QD_DEV void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// 32 TMEM lanes x 64 columns of 32 bits for this warp.
QD_DEV void tmem_ld_32x64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Eight Q8_0 weights (two 32-bit words of int8) -> four bf16 pairs, each
// bf16(f32(d) * q). q + 128 is placed in the low mantissa bits of 2^23 and the
// bias subtracted, which gives q exactly; q * d is exact in binary32 (8 by 11
// significant bits), so the pack's round to nearest even is the only rounding.
QD_DEV uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
QD_DEV uint4 widen8_q8(uint32_t w0, uint32_t w1, float d) {
  uint32_t o[4];
  const uint32_t u[2] = {w0 ^ 0x80808080u, w1 ^ 0x80808080u};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float f[4];
#pragma unroll
    for (int b = 0; b < 4; ++b)
      f[b] = (__uint_as_float(__byte_perm(u[h], 0x4B000000u, 0x7540u + b)) - 8388736.0f) * d;
    o[2 * h] = bf16x2_bits(f[0], f[1]);
    o[2 * h + 1] = bf16x2_bits(f[2], f[3]);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Ring depths of the Q8_0 form (one CTA per SM, ~216 KB of shared memory). The
// converters work as kConvGroups groups of two warps, group g widening K steps
// g, g + kConvGroups, ...: a single step's widening is a chain of loads, math,
// stores and a proxy fence whose latency one group alone cannot hide, so several
// steps are widened at once. The A ring holds those steps plus the MMA's; the
// int8 ring carries the HBM stream (about 68 KB in flight per SM); X comes from L2.
constexpr int kConvGroups = kConvWarps / 2;
constexpr int kQSt = 8;    // int8 + scale tiles
constexpr int kBSt = 5;    // X tiles
constexpr int kASt = 6;    // widened bf16 A tiles

// Bounded wait for the last copy issued to each slot of a ring (a CTA never
// exits with a TMA copy still landing in its shared memory).
QD_DEV void drain_ring(uint64_t* full, int slots, int issued, int* err) {
  for (int i = max(0, issued - slots); i < issued; ++i) mbar_wait_bounded(&full[i % slots], (uint32_t)((i / slots) & 1), err);
}

// BN: tokens per CTA (the MMA's N and the TMEM columns): 64, or 256 for many rows
template <int kStagesTc, bool kQ8, int BN>
__global__ void __launch_bounds__(kQ8 ? kThreadsQ8 : kThreadsTc, (!kQ8 && kStagesTc <= 3 && BN == kBN) ? 3 : 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmS, const TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  constexpr int nA = kQ8 ? kASt : kStagesTc;  // A tiles (bf16 W, or widened Q8_0)
  constexpr int nB = kQ8 ? kBSt : kStagesTc;  // X tiles
  constexpr int nQ = kQ8 ? kQSt : 0;          // int8 + scale tiles
  constexpr int kTileB = BN * kBK * 2;        // X tile bytes
  unsigned char* sA = smem;                   // [nA][128 x 128 B]
  unsigned char* sB = sA + nA * kTileA;       // [nB][BN x 128 B]
  unsigned char* sQ = sB + nB * kTileB;       // [nQ][128 x 64 B]
  unsigned char* sS = sQ + nQ * kTileQ;       // [nQ][128 x 16 B]
  // bf16 form: full/empty per stage cover both A and B tiles
  uint64_t* full = (uint64_t*)(sS + nQ * kTileS);   // [nA] A+B landed / [nB] X landed (Q8_0)
  uint64_t* empty = full + nB;                      // [nB] stage read by the MMA
  uint64_t* qfull = empty + nB;                     // [nQ] int8 + scales landed
  uint64_t* qempty = qfull + nQ;                    // [nQ] int8 tile read by the converters
  uint64_t* conv = qempty + nQ;                     // [nA] A tile widened (Q8_0)
  uint64_t* aempty = conv + (kQ8 ? nA : 0);         // [nA] A tile read by the MMA (Q8_0)
  uint64_t* done = aempty + (kQ8 ? nA : 0);
  uint32_t* tmem_slot = (uint32_t*)(done + 1);
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = (p.zfast ? blockIdx.y : blockIdx.x) * kBM;
  const int n0 = (p.zfast ? blockIdx.x : blockIdx.z) * BN;   // this CTA's first token
  // this CTA's K blocks [kb0, kb0 + n_k) of its split (grid y unless token tiles lead)
  const int split = p.zfast ? 0 : (int)blockIdx.y;
  const int n_kt = p.K / kBK;
  const int kb0 = (int)(((long long)n_kt * split) / p.splits);
  const int n_k = (int)(((long long)n_kt * (split + 1)) / p.splits) - kb0;
  __shared__ int s_ticket;

  if (tid == 0) {
    for (int i = 0; i < nB; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < nQ; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 2);  // the two warps of the step's converter group
    }
    if (kQ8)
      for (int i = 0; i < nA; ++i) {
        mbar_init(&conv[i], 2);
        mbar_init(&aempty[i], 1);
      }
    mbar_init(done, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(tmem_slot, BN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  auto mma_stage = [&](uint32_t a0, uint32_t b0, int i) {
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk)
      mma_bf16<BN>(tmem, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), (i | kk) != 0);
  };

  if constexpr (!kQ8) {
    if (warp == 0 && lane == 0) {
      // ---- producer: W tiles need no dependency; X (this step's activations) does
      const int pre = min(kStagesTc, n_k);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], kTileA + kTileB);
        tma_load_2d(sA + i * kTileA, &tmW, (kb0 + i) * kBK, row0, &full[i]);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) tma_load_2d(sB + i * kTileB, &tmX, (kb0 + i) * kBK, n0, &full[i]);
      int issued = pre;
      for (int i = pre; i < n_k; ++i) {
        const int s = i % kStagesTc;
        if (!mbar_wait_bounded(&empty[s], (uint32_t)(((i / kStagesTc) - 1) & 1), p.err)) {
          s_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kTileA + kTileB);
        tma_load_2d(sA + s * kTileA, &tmW, (kb0 + i) * kBK, row0, &full[s]);
        tma_load_2d(sB + s * kTileB, &tmX, (kb0 + i) * kBK, n0, &full[s]);
        issued = i + 1;
      }
      drain_ring(full, kStagesTc, issued, p.err);
    } else if (warp == 1 && lane == 0) {
      // ---- MMA issuer
      for (int i = 0; i < n_k; ++i) {
        const int s = i % kStagesTc;
        if (!mbar_wait_bounded(&full[s], (uint32_t)((i / kStagesTc) & 1), p.err)) {
          s_abort = 1;  // D holds a partial sum: the epilogue must not store it
          break;
        }
        tc_fence_after();
        mma_stage(smem_u32(sA + s * kTileA), smem_u32(sB + s * kTileB), i);
        mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
      }
      mma_commit(done);         // D complete (also arrives after an early exit)
    }
  } else {
    if (warp == 0 && lane == 0) {
      // ---- weight producer: int8 tiles and their scales (no dependency on the
      // previous kernel), as far ahead as the int8 ring allows
      int issued = 0;
      for (int i = 0; i < n_k; ++i) {
        const int s = i % kQSt;
        if (i >= kQSt && !mbar_wait_bounded(&qempty[s], (uint32_t)(((i / kQSt) - 1) & 1), p.err)) {
          s_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&qfull[s], kTileQ + kTileS);
        tma_load_2d(sQ + s * kTileQ, &tmW, (kb0 + i) * kBK, row0, &qfull[s]);
        tma_load_2d(sS + s * kTileS, &tmS, ((kb0 + i) >> 2) * 8, row0, &qfull[s]);  // 16-byte aligned x
        issued = i + 1;
      }
      drain_ring(qfull, kQSt, issued, p.err);
    } else if (warp == 2 && lane == 0) {
      // ---- activation producer: this step's X tiles (from L2)
      pdl_wait();
      int issued = 0;
      for (int i = 0; i < n_k; ++i) {
        const int s = i % kBSt;
        if (i >= kBSt && !mbar_wait_bounded(&empty[s], (uint32_t)(((i / kBSt) - 1) & 1), p.err)) {
          s_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kTileB);
        tma_load_2d(sB + s * kTileB, &tmX, (kb0 + i) * kBK, n0, &full[s]);
        issued = i + 1;
      }
      drain_ring(full, kBSt, issued, p.err);
    } else if (warp == 1 && lane == 0) {
      // ---- MMA issuer
      for (int i = 0; i < n_k; ++i) {
        const int sa = i % kASt, sb = i % kBSt;
        if (!mbar_wait_bounded(&full[sb], (uint32_t)((i / kBSt) & 1), p.err) ||
            !mbar_wait_bounded(&conv[sa], (uint32_t)((i / kASt) & 1), p.err)) {
          s_abort = 1;
          break;
        }
        tc_fence_after();
        mma_stage(smem_u32(sA + sa * kTileA), smem_u32(sB + sb * kTileB), i);
        mma_commit(&aempty[sa]);
        mma_commit(&empty[sb]);
      }
      mma_commit(done);
    } else if (warp >= 4) {
      // ---- converters: int8 tile + scales -> bf16 A tile in the 128-byte-swizzle
      // layout TMA would have written (16-byte chunk c of row r at chunk c ^ (r & 7)).
      // In a group, thread t (0..63) takes 16 int8 of a row per item: rows t / 4 + 16 j
      // (j < 8), chunk t % 4, so a warp reads 512 contiguous bytes per j and its
      // swizzled stores hit distinct banks. All eight items are loaded before the
      // int8 slot is released, then widened and stored.
      const int grp = (warp - 4) >> 1;
      const int t = ((warp - 4) & 1) * 32 + lane;
      for (int i = grp; i < n_k; i += kConvGroups) {
        const int sq = i % kQSt, sa = i % kASt;
        if (!mbar_wait_bounded(&qfull[sq], (uint32_t)((i / kQSt) & 1), p.err) ||
            (i >= kASt && !mbar_wait_bounded(&aempty[sa], (uint32_t)(((i / kASt) - 1) & 1), p.err))) {
          s_abort = 1;
          break;
        }
        const int kt = kb0 + i;
        const unsigned char* q = sQ + sq * kTileQ;
        const __half* sc = (const __half*)(sS + sq * kTileS);
        const int c = t & 3, r0 = t >> 2;
        uint4 w[8];
        float d[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int row = r0 + 16 * j;
          w[j] = *(const uint4*)(q + row * kBK + c * 16);
          d[j] = __half2float(sc[row * 8 + (kt & 3) * 2 + (c >> 1)]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[sq]);
        unsigned char* a = sA + sa * kTileA;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int row = r0 + 16 * j, sw = row & 7;
          *(uint4*)(a + row * 128 + (((2 * c) ^ sw) << 4)) = widen8_q8(w[j].x, w[j].y, d[j]);
          *(uint4*)(a + row * 128 + (((2 * c + 1) ^ sw) << 4)) = widen8_q8(w[j].z, w[j].w, d[j]);
        }
        fence_proxy_async_smem();  // the generic-proxy stores before the MMA's reads
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv[sa]);
      }
    }
  }
  __syncwarp();
  // every role has left its loop: an abort flag set by any of them is visible below
  __syncthreads();

  // ---- epilogue: warp w < 4 owns TMEM lanes [32w, 32w + 32) = rows row0 + 32w + lane
  pdl_wait();
  const bool rows_here = !kQ8 || warp < 4;
  const bool ok = rows_here ? mbar_wait_bounded(done, 0, p.err) : true;
  tc_fence_after();
  float v[64];
  if (rows_here) tmem_ld_32x64(tmem + ((uint32_t)(warp * 32) << 16), v);
  const int rl = warp * 32 + lane;          // this thread's row of the tile
  const int r = row0 + rl;
  bool write = rows_here && ok && !s_abort;
  // y[t + j, r] (+)= o[j] for 16 tokens from t; the residual values are all loaded
  // before any store, so the 16 read-modify-writes overlap instead of queueing
  auto store_rows = [&](int t, const float* o) {
    float old[16];
    if (p.epi == EPI_RESID_ADD) {
#pragma unroll
      for (int j = 0; j < 16; ++j) old[j] = t + j < p.B ? p.y[(size_t)(t + j) * p.R + r] : 0.f;
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) old[j] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (t + j < p.B) p.y[(size_t)(t + j) * p.R + r] = p.epi == EPI_RESID_ADD ? old[j] + o[j] : o[j];
  };
  if (p.splits > 1) {
    // publish this split's partial tile [kBN tokens][kBM rows] (each warp access
    // one 128-byte line), take a ticket; the last split of the tile adds every
    // partial in split order, 16 tokens at a time with all their loads (and the
    // residual's) in flight together
    const size_t tile = blockIdx.x;
    float* part = p.part + (tile * p.splits + split) * (size_t)(kBN * kBM);
    if (rows_here) {
#pragma unroll
      for (int n = 0; n < kBN; ++n) part[(size_t)n * kBM + rl] = v[n];
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      s_ticket = atomicAdd(p.cnt + tile, 1);
      __threadfence();
    }
    __syncthreads();
    if (s_ticket == p.splits - 1 && write && r < p.R) {
      const float* base = p.part + tile * p.splits * (size_t)(kBN * kBM) + rl;
      const bool radd = p.epi == EPI_RESID_ADD;
#pragma unroll 1
      for (int c = 0; c < kBN / 16; ++c) {
        float t[kMaxSplits][16], yo[16];
#pragma unroll
        for (int sp = 0; sp < kMaxSplits; ++sp)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            t[sp][j] = sp < p.splits ? __ldcg(base + ((size_t)sp * kBN + c * 16 + j) * kBM) : 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          yo[j] = (radd && c * 16 + j < p.B) ? p.y[(size_t)(c * 16 + j) * p.R + r] : 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float a = t[0][j];
#pragma unroll
          for (int sp = 1; sp < kMaxSplits; ++sp)
            if (sp < p.splits) a += t[sp][j];
          if (c * 16 + j < p.B) p.y[(size_t)(c * 16 + j) * p.R + r] = radd ? yo[j] + a : a;
        }
      }
    }
    if (s_ticket == p.splits - 1 && tid == 0) p.cnt[tile] = 0;
    write = false;  // the tile's output is written above (or by another split)
  }
  if (p.splits <= 1 && rows_here) {
    // 64 TMEM columns (tokens) at a time; the loads are warp-wide, the stores per row
#pragma unroll 1
    for (int c4 = 0; c4 < BN / 64; ++c4) {
      if (c4 > 0) tmem_ld_32x64(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c4 * 64), v);
      if (write && r < p.R) {
#pragma unroll
        for (int c = 0; c < 4; ++c) store_rows(n0 + c4 * 64 + c * 16, v + c * 16);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, BN);
}

// ---- persistent wide form (many token rows, bf16 weights) ----------------------
// One CTA per SM loops over (128-row weight tile, 256-token tile) items, the token
// tiles of a weight tile consecutive (they share it through L2). Warp 0 streams the
// W and X boxes through a 4-stage ring, warp 1 issues the MMAs into one of two
// 256-column TMEM accumulators, and warps 2..5 drain the other one to y (warp w
// reads TMEM lane quarter w % 4), so one tile's epilogue runs under the next tile's
// MMAs instead of leaving the tensor pipe idle while the SM's next CTA refills its ring.
constexpr int kWdSt = 4;
constexpr int kWdBN = 256;
constexpr int kWdTileX = kWdBN * kBK * 2;   // 32 KB
constexpr int kWdThreads = 192;
constexpr int kWdXch = 2 * 2 * 64 * 32 * 4;   // SwiGLU form: [2 lane pairs][2 buffers][64 columns][32 lanes] f32
// shared memory: ring, (SwiGLU) exchange buffers, then the barriers
__host__ __device__ constexpr size_t wd_smem(bool sw) {
  return 1024 + (size_t)kWdSt * (kTileA + kWdTileX) + (sw ? kWdXch : 0) + (2 * kWdSt + 4 + 8) * 8 + 16;
}

// kSw = false: y[t, r] (+)= sum_k W[r, k] X[t, k], weight tiles of 128 rows.
// kSw = true (the gate+up projection with SwiGLU): a weight tile is gate rows
// j0 .. j0 + 63 (TMEM lanes 0..63) over up rows F + j0 .. (lanes 64..127), two 64-row
// boxes per stage, so one M = 128 x N = 256 accumulator covers 64 outputs of h and two
// accumulators still fit in TMEM. The up warps (lane quarters 2, 3) hand their values
// to the gate warps (quarters 0, 1) through shared memory, 64 columns at a time, and
// the gate warps write h[t, j] = bf16(silu(g) u) with the SwiGLU rows kernel's arithmetic.
template <bool kSw>
__global__ void __launch_bounds__(kWdThreads, 1) gemm_wide_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                   const __grid_constant__ CUtensorMap tmX,
                                                                   const TcParams p, __nv_bfloat16* h, int F) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sA = smem;                              // [kWdSt][128 x 128 B]
  unsigned char* sB = sA + kWdSt * kTileA;               // [kWdSt][256 x 128 B]
  float* xch = (float*)(sB + kWdSt * kWdTileX);          // kSw: [pair][buf][64][32]
  uint64_t* full = (uint64_t*)((unsigned char*)xch + (kSw ? kWdXch : 0));   // [kWdSt] W and X boxes landed
  uint64_t* empty = full + kWdSt;                        // [kWdSt] the stage's MMAs are done
  uint64_t* acc_full = empty + kWdSt;                    // [2] an accumulator holds a finished tile
  uint64_t* acc_empty = acc_full + 2;                    // [2] the epilogue drained it (4 warps)
  uint64_t* xfull = acc_empty + 2;                       // kSw: [pair * 2 + buf] up values written (32 lanes)
  uint64_t* xempty = xfull + 4;                          // kSw: [pair * 2 + buf] up values read (32 lanes)
  uint32_t* tmem_slot = (uint32_t*)(xempty + 4);
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_kt = p.K / kBK;
  const int NT = (p.B + kWdBN - 1) / kWdBN;
  constexpr int kRows = kSw ? kBM / 2 : kBM;   // output rows per weight tile
  const int items = (((kSw ? F : p.R) + kRows - 1) / kRows) * NT;
  if (tid == 0) {
    for (int i = 0; i < kWdSt; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&xfull[i], 32);
      mbar_init(&xempty[i], 32);
    }
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 1) tmem_alloc(tmem_slot, 2 * kWdBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {  // ---- producer: W boxes need no dependency, X boxes (activations) do
      int it = 0, issued = 0;
      bool waited = false, ok = true;
      for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
        const int rt = item / NT, nt = item - rt * NT;
        for (int kb = 0; kb < n_kt; ++kb, ++it) {
          const int st = it % kWdSt;
          if (it >= kWdSt && !mbar_wait_bounded(&empty[st], (uint32_t)(((it / kWdSt) - 1) & 1), p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], kTileA + kWdTileX);
          if (kSw) {
            tma_load_2d(sA + st * kTileA, &tmW, kb * kBK, rt * kRows, &full[st]);
            tma_load_2d(sA + st * kTileA + kTileA / 2, &tmW, kb * kBK, F + rt * kRows, &full[st]);
          } else {
            tma_load_2d(sA + st * kTileA, &tmW, kb * kBK, rt * kBM, &full[st]);
          }
          if (!waited) {
            pdl_wait();
            waited = true;
          }
          tma_load_2d(sB + st * kWdTileX, &tmX, kb * kBK, nt * kWdBN, &full[st]);
          issued = it + 1;
        }
      }
      if (!ok) *(volatile int*)&s_abort = 1;
      drain_ring(full, kWdSt, issued, p.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer
      int it = 0, j = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++j) {
        const int a = j & 1;
        if (j >= 2 && !mbar_wait_bounded(&acc_empty[a], (uint32_t)(((j >> 1) - 1) & 1), p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(a * kWdBN);
        for (int kb = 0; kb < n_kt; ++kb, ++it) {
          const int st = it % kWdSt;
          if (!mbar_wait_bounded(&full[st], (uint32_t)((it / kWdSt) & 1), p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + st * kTileA), b0 = smem_u32(sB + st * kWdTileX);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16<kWdBN>(d, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), (kb | kk) != 0);
          mma_commit(&empty[st]);
        }
        if (!ok) break;
        mma_commit(&acc_full[a]);
      }
      if (!ok) *(volatile int*)&s_abort = 1;
    }
  } else {
    // ---- epilogue warps 2..5: TMEM lane quarter q = warp % 4, rows 32 q + lane of a tile
    pdl_wait();   // y (the residual stream) comes from earlier kernels
    const int q = warp & 3;
    const uint32_t lanes = (uint32_t)(q * 32) << 16;
    const int pair = q & 1;   // kSw: gate quarter `pair` takes the values of up quarter 2 + pair
    const bool up = q >= 2;
    float v[64];
    int j = 0, xc = 0;
    bool live = true;
    for (int item = blockIdx.x; item < items && live; item += gridDim.x, ++j) {
      const int a = j & 1;
      const bool got = mbar_wait_bounded(&acc_full[a], (uint32_t)((j >> 1) & 1), p.err) && !*(volatile int*)&s_abort;
      if (!__all_sync(0xffffffffu, got)) break;   // warp-wide TMEM loads: one decision per warp
      tc_fence_after();
      const int rt = item / NT, nt = item - rt * NT;
      const int n0 = nt * kWdBN;
      if (kSw) {
        const int jr = rt * kRows + pair * 32 + lane;   // the h column of this lane (gate warps)
#pragma unroll 1
        for (int c4 = 0; c4 < kWdBN / 64; ++c4, ++xc) {
          tmem_ld_32x64(tmem + lanes + (uint32_t)(a * kWdBN + c4 * 64), v);
          const int bsel = pair * 2 + (xc & 1), use = xc >> 1;
          float* xb = xch + bsel * (64 * 32);
          if (up) {
            const bool free_ = use == 0 || mbar_wait_bounded(&xempty[bsel], (uint32_t)((use - 1) & 1), p.err);
            if (!__all_sync(0xffffffffu, free_)) {
              live = false;
              break;
            }
#pragma unroll
            for (int c = 0; c < 64; ++c) xb[c * 32 + lane] = v[c];
            mbar_arrive(&xfull[bsel]);
          } else {
            const bool ready = mbar_wait_bounded(&xfull[bsel], (uint32_t)(use & 1), p.err);
            if (!__all_sync(0xffffffffu, ready)) {
              live = false;
              break;
            }
#pragma unroll
            for (int c = 0; c < 64; ++c) v[c] = v[c] / (1.0f + expf(-v[c])) * xb[c * 32 + lane];
            mbar_arrive(&xempty[bsel]);
            if (jr < F) {
#pragma unroll
              for (int c = 0; c < 64; ++c) {
                const int n = n0 + c4 * 64 + c;
                if (n < p.B) h[(size_t)n * F + jr] = __float2bfloat16_rn(v[c]);
              }
            }
          }
        }
        if (!live) {
          *(volatile int*)&s_abort = 1;
          break;
        }
      } else {
        const int r = rt * kBM + q * 32 + lane;
        // y[t + j, r] (+)= o[j] for 16 tokens from t, the residual values loaded first
        auto store_rows = [&](int t, const float* o) {
          float old[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            old[e] = (p.epi == EPI_RESID_ADD && t + e < p.B) ? p.y[(size_t)(t + e) * p.R + r] : 0.f;
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (t + e < p.B) p.y[(size_t)(t + e) * p.R + r] = p.epi == EPI_RESID_ADD ? old[e] + o[e] : o[e];
        };
#pragma unroll 1
        for (int c4 = 0; c4 < kWdBN / 64; ++c4) {
          tmem_ld_32x64(tmem + lanes + (uint32_t)(a * kWdBN + c4 * 64), v);
          if (r < p.R && n0 + c4 * 64 < p.B) {
#pragma unroll
            for (int c = 0; c < 4; ++c) store_rows(n0 + c4 * 64 + c * 16, v + c * 16);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kWdBN);
  }
}

// QD_GEMM_WIDE (read per call): the many-row bf16 GEMMs run on the persistent form
// above (24576 x 4096 weights x 2048 tokens: 262 us against 285 us for one CTA per
// tile); "tiles" keeps one CTA per 128 x 256 tile.
bool gemm_wide_persistent() {
  const char* v = getenv("QD_GEMM_WIDE");
  return !(v && strcmp(v, "tiles") == 0);
}

cudaError_t launch_wide(const CUtensorMap& tw, const CUtensorMap& tx, const TcParams& p, const Launch& L) {
  const int items = ((p.R + kBM - 1) / kBM) * ((p.B + kWdBN - 1) / kWdBN);
  const int grid = std::min(items, dev_info().sm_count);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_wide_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wd_smem(false));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(gemm_wide_kernel<false>, dim3(grid), dim3(kWdThreads), wd_smem(false), L, tw, tx, p,
                   (__nv_bfloat16*)nullptr, 0);
}

// ---- prefill gate+up with SwiGLU in the epilogue ------------------------------
// The gate rows j0 .. j0 + 127 and the up rows F + j0 .. of W_gu against one
// 256-token tile of X: two M = 128 x N = 256 accumulators (all 512 TMEM
// columns), each stage bringing the gate box, the up box and the X box. The
// epilogue writes h[t, j] = bf16(silu(g) * u) straight from the accumulators, the
// arithmetic of the SwiGLU rows kernel, so the f32 [gate; up] rows never reach
// memory.
constexpr int kSwBN = 256;
constexpr int kSwSt = 3;
constexpr int kTileX256 = kSwBN * kBK * 2;   // 32 KB

struct SwParams {
  int F, K, B;
  __nv_bfloat16* h;   // [B, F]
  int* err;
};

// 32 TMEM lanes x 32 columns of 32 bits for this warp.
QD_DEV void tmem_ld_32x32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kThreadsTc, 1)
    gemm_tc_swiglu_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                          const SwParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sG = smem;                          // [kSwSt][128 x 128 B] gate rows
  unsigned char* sU = sG + kSwSt * kTileA;           // [kSwSt][128 x 128 B] up rows
  unsigned char* sB = sU + kSwSt * kTileA;           // [kSwSt][256 x 128 B] X rows
  uint64_t* full = (uint64_t*)(sB + kSwSt * kTileX256);
  uint64_t* empty = full + kSwSt;
  uint64_t* done = empty + kSwSt;
  uint32_t* tmem_slot = (uint32_t*)(done + 1);
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j0 = blockIdx.y * kBM;        // gate rows j0 .., up rows F + j0 ..
  const int n0 = blockIdx.x * kSwBN;      // tokens n0 ..
  const int n_k = p.K / kBK;
  if (tid == 0) {
    for (int i = 0; i < kSwSt; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0 && lane == 0) {
    // ---- producer: the weight boxes of the first stages go out before the dependency wait
    const int pre = min(kSwSt, n_k);
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&full[i], 2 * kTileA + kTileX256);
      tma_load_2d(sG + i * kTileA, &tmW, i * kBK, j0, &full[i]);
      tma_load_2d(sU + i * kTileA, &tmW, i * kBK, p.F + j0, &full[i]);
    }
    pdl_wait();
    for (int i = 0; i < pre; ++i) tma_load_2d(sB + i * kTileX256, &tmX, i * kBK, n0, &full[i]);
    int issued = pre;
    for (int i = pre; i < n_k; ++i) {
      const int s = i % kSwSt;
      if (!mbar_wait_bounded(&empty[s], (uint32_t)(((i / kSwSt) - 1) & 1), p.err)) {
        s_abort = 1;
        break;
      }
      mbar_arrive_expect_tx(&full[s], 2 * kTileA + kTileX256);
      tma_load_2d(sG + s * kTileA, &tmW, i * kBK, j0, &full[s]);
      tma_load_2d(sU + s * kTileA, &tmW, i * kBK, p.F + j0, &full[s]);
      tma_load_2d(sB + s * kTileX256, &tmX, i * kBK, n0, &full[s]);
      issued = i + 1;
    }
    drain_ring(full, kSwSt, issued, p.err);
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: gate into TMEM columns 0 .. 255, up into 256 .. 511
    for (int i = 0; i < n_k; ++i) {
      const int s = i % kSwSt;
      if (!mbar_wait_bounded(&full[s], (uint32_t)((i / kSwSt) & 1), p.err)) {
        s_abort = 1;
        break;
      }
      tc_fence_after();
      const uint32_t g0 = smem_u32(sG + s * kTileA), u0 = smem_u32(sU + s * kTileA), b0 = smem_u32(sB + s * kTileX256);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        mma_bf16<kSwBN>(tmem, smem_desc_sw128(g0 + kk * 32), smem_desc_sw128(b0 + kk * 32), (i | kk) != 0);
        mma_bf16<kSwBN>(tmem + kSwBN, smem_desc_sw128(u0 + kk * 32), smem_desc_sw128(b0 + kk * 32), (i | kk) != 0);
      }
      mma_commit(&empty[s]);
    }
    mma_commit(done);
  }
  __syncwarp();
  __syncthreads();

  // ---- epilogue: warp w owns TMEM lanes 32w .. 32w + 31 = gate/up rows j0 + 32w + lane
  pdl_wait();
  const bool ok = mbar_wait_bounded(done, 0, p.err);
  tc_fence_after();
  const int j = j0 + warp * 32 + lane;
  const bool write = ok && !s_abort && j < p.F;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
  for (int c = 0; c < kSwBN / 32; ++c) {
    float g[32], u[32];
    tmem_ld_32x32(tmem + lane_off + (uint32_t)(c * 32), g);
    tmem_ld_32x32(tmem + lane_off + (uint32_t)(kSwBN + c * 32), u);
    if (write) {
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int n = n0 + c * 32 + t;
        if (n < p.B) p.h[(size_t)n * p.F + j] = __float2bfloat16_rn(g[t] / (1.0f + expf(-g[t])) * u[t]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// --- host: tensor maps --------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  });
  return fn;
}

// Row-major [rows, cols] matrix of elem-byte elements, box of box_rows x box_cols.
cudaError_t encode_rowmajor(CUtensorMap* m, CUtensorMapDataType dt, int elem, const void* base, uint64_t rows,
                            uint64_t cols, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * elem};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Row-major bf16 [rows, cols] matrix, box of box_rows x 64 columns, 128-byte swizzle.
cudaError_t encode_rowmajor_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                                 uint32_t box_rows) {
  return encode_rowmajor(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, kBK, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

constexpr size_t smem_tc(int st, bool q8, int bn) {
  return q8 ? 1024 + (size_t)kASt * kTileA + (size_t)kBSt * bn * kBK * 2 + (size_t)kQSt * (kTileQ + kTileS) +
                  (2 * kBSt + 2 * kQSt + 2 * kASt + 1) * 8 + 16
            : 1024 + (size_t)st * (kTileA + (size_t)bn * kBK * 2) + (2 * st + 1) * 8 + 16;
}

template <int ST, bool Q8, int BN = kBN>
cudaError_t launch_tc(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& ts, const TcParams& p,
                      int tiles, const Launch& L) {
  auto k = gemm_tc_kernel<ST, Q8, BN>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_tc(ST, Q8, BN));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const dim3 grid = p.zfast ? dim3(ceil_div(p.B, BN), tiles) : dim3(tiles, p.splits, ceil_div(p.B, BN));
  return launch_ex(k, grid, dim3(Q8 ? kThreadsQ8 : kThreadsTc), smem_tc(ST, Q8, BN), L, tw, tx, ts, p);
}

}  // namespace

cudaError_t encode_tmap_bf16_2d(void* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return encode_rowmajor_bf16((CUtensorMap*)map, base, rows, cols, box_rows);
}

cudaError_t encode_tmap_u8_sw128(void* map, const void* base, uint64_t rows, uint64_t cols_bytes, uint32_t box_rows) {
  return encode_rowmajor((CUtensorMap*)map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, cols_bytes, 128, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

bool gemm_tc_supported(int R, int K, int B) { return R >= 1 && K >= kBK && K % kBK == 0 && B >= 1 && B <= kBN; }

// Many rows (prefill): 64-token tiles over grid z, no K split.
bool gemm_tc_rows_supported(int R, int K, int B, bool q8) {
  return R >= 1 && K >= kBK && K % kBK == 0 && (!q8 || K % 256 == 0) && B >= 1 && B <= 65535 * kBN;
}

// Q8_0 weights: the scale rows are read as 16-byte TMA boxes (256 columns), so
// their stride K/32 x 2 bytes must be a multiple of 16.
bool gemm_tc_q8_supported(int R, int K, int B) { return gemm_tc_supported(R, K, B) && K % 256 == 0; }

// K splits for an R x K launch, chosen to keep every SM streaming to the end.
// With s splits the tiles x s CTAs run in ceil(tiles x s / SMs) rounds of 1/s of
// a tile's weight bytes each; every split adds a 32 KB partial tile written and
// read back (mostly through L2, counted at half weight). At least 8 K blocks per
// CTA, at most kMaxSplits. QD_GEMM_SPLITS forces a count.
// Split-K workspace: a fixed block of tile tickets first (the same place for every
// launch that shares the workspace, so one launch's partials never land on
// another's tickets), then the partial tiles.
constexpr int kMaxSplitTiles = 4096;
constexpr size_t kTicketBytes = (size_t)kMaxSplitTiles * sizeof(int);

int gemm_tc_splits(int R, int K, bool q8) {
  if (R < 1 || K < kBK) return 1;
  const int tiles = (R + kBM - 1) / kBM, n_kt = K / kBK, sms = dev_info().sm_count;
  if (tiles > kMaxSplitTiles) return 1;
  static const int forced = [] {
    const char* v = getenv("QD_GEMM_SPLITS");
    return v ? atoi(v) : 0;
  }();
  if (forced > 0) return std::max(1, std::min(std::min(forced, kMaxSplits), n_kt));
  // bf16: two or three CTAs per SM, so tiles that fill the SMs are not split (measured
  // slower); Q8_0 runs one CTA per SM, where splitting evens out a partial last wave
  if (tiles >= sms && !q8) return 1;
  int best = 1;
  double best_t = (double)((tiles + sms - 1) / sms);
  const double tile_bytes = (double)kBM * K * (q8 ? 34.0 / 32.0 : 2.0);
  for (int sp = 2; sp <= kMaxSplits && n_kt / sp >= 8; ++sp) {
    const double t = (double)((tiles * sp + sms - 1) / sms) / sp + 0.5 * sp * 65536.0 / tile_bytes;
    if (t < best_t) {
      best_t = t;
      best = sp;
    }
  }
  return best;
}

size_t gemm_tc_workspace_bytes(int R, int K, bool q8) {
  const int sp = gemm_tc_splits(R, K, q8);
  if (sp <= 1) return 0;
  const size_t tiles = (size_t)(R + kBM - 1) / kBM;
  return kTicketBytes + tiles * sp * kBN * kBM * sizeof(float);
}

cudaError_t launch_gemm_tc(const GemmTcArgs& a, const Launch& L) {
  const bool q8 = a.S != nullptr;
  const bool rows = a.B > kBN;   // several token tiles: no K split
  if (rows ? !gemm_tc_rows_supported(a.R, a.K, a.B, q8)
           : !(q8 ? gemm_tc_q8_supported(a.R, a.K, a.B) : gemm_tc_supported(a.R, a.K, a.B)))
    return cudaErrorInvalidValue;
  CUtensorMap tw, tx, ts;
  cudaError_t e;
  if (q8) {
    // int8 [R, K] in 128 x 64-byte boxes; fp16 scales [R, K/32] in 128 x 8 boxes;
    // rows past R read as zeros
    e = encode_rowmajor(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.W, (uint64_t)a.R, (uint64_t)a.K, kBK, kBM,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    e = encode_rowmajor(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.S, (uint64_t)a.R, (uint64_t)a.K / 32, 8, kBM,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    e = encode_rowmajor_bf16(&tw, a.W, (uint64_t)a.R, (uint64_t)a.K, kBM);
    ts = tw;  // unused
  }
  if (e != cudaSuccess) return e;
  // many rows (bf16): 256-token tiles (QD_GEMM_BN=64 keeps 64)
  static const int forced_bn = [] {
    const char* v = getenv("QD_GEMM_BN");
    return v ? atoi(v) : 0;
  }();
  const bool wide = !q8 && rows && a.B > 2 * kBN && forced_bn != kBN;
  // X has B rows; the box reads zeros past them
  e = encode_rowmajor_bf16(&tx, a.X, (uint64_t)a.B, (uint64_t)a.K, wide ? 256 : kBN);
  if (e != cudaSuccess) return e;
  TcParams p = {};
  p.R = a.R; p.K = a.K; p.B = a.B; p.epi = a.epi; p.y = a.y; p.err = L.err;
  p.zfast = rows ? 1 : 0;
  const int tiles = (a.R + kBM - 1) / kBM;
  p.splits = 1;
  const size_t need = gemm_tc_workspace_bytes(a.R, a.K, q8);
  if (!rows && a.ws && need > 0 && a.ws_bytes >= need) {
    p.splits = gemm_tc_splits(a.R, a.K, q8);
    p.cnt = (int*)a.ws;
    p.part = (float*)((unsigned char*)a.ws + kTicketBytes);
  }
  // Q8_0: one 384-thread CTA per SM with its own ring depths
  if (q8) return launch_tc<kASt, true>(tw, tx, ts, p, tiles, L);
  if (wide) return gemm_wide_persistent() ? launch_wide(tw, tx, p, L) : launch_tc<4, false, 256>(tw, tx, ts, p, tiles, L);
  static const int forced = [] {
    const char* v = getenv("QD_GEMM_STAGES");
    return v ? atoi(v) : 0;
  }();
  const bool deep =
      forced == 6 || (forced != 3 && (long long)tiles * p.splits * ceil_div(a.B, kBN) <= dev_info().sm_count);
  return deep ? launch_tc<6, false>(tw, tx, ts, p, tiles, L) : launch_tc<3, false>(tw, tx, ts, p, tiles, L);
}

// ---- Q8_0 weights widened to bf16 for the prefill's many-row GEMMs ---------
// out[r, k] = bf16(f32(d) * q) for every weight of a Q8_0 matrix (int8 [R, K], fp16
// scales [R, K / 32]), the converters' arithmetic above, one 32-weight block per thread
// per grid-stride step. The stores wait for the kernels before this one, which may still
// read the output buffer.
__global__ void __launch_bounds__(256) q8_widen_kernel(const uint4* __restrict__ q, const __half* __restrict__ sc,
                                                       uint4* __restrict__ out, size_t n_blocks) {
  pdl_wait();
  pdl_launch_dependents();
  for (size_t b = (size_t)blockIdx.x * blockDim.x + threadIdx.x; b < n_blocks; b += (size_t)gridDim.x * blockDim.x) {
    const uint4 w0 = __ldg(q + 2 * b), w1 = __ldg(q + 2 * b + 1);
    const float d = __half2float(sc[b]);
    out[4 * b] = widen8_q8(w0.x, w0.y, d);
    out[4 * b + 1] = widen8_q8(w0.z, w0.w, d);
    out[4 * b + 2] = widen8_q8(w1.x, w1.y, d);
    out[4 * b + 3] = widen8_q8(w1.z, w1.w, d);
  }
}

cudaError_t launch_q8_widen(const void* W, const void* S, int R, int K, void* out, const Launch& L) {
  if (R < 1 || K < 32 || K % 32 != 0 || !W || !S || !out || ((uintptr_t)W & 15) || ((uintptr_t)out & 15))
    return cudaErrorInvalidValue;
  const size_t n_blocks = (size_t)R * (K / 32);
  const int grid = (int)std::min<size_t>((n_blocks + 255) / 256, (size_t)dev_info().sm_count * 8);
  return launch_ex(q8_widen_kernel, dim3(grid), dim3(256), 0, L, (const uint4*)W, (const __half*)S, (uint4*)out,
                   n_blocks);
}

// From 1024 rows: below that the paired tiles (one CTA per SM for their shared
// memory) leave too few CTAs to balance the SMs (512 rows measured 4 % slower than
// the GEMM + SwiGLU rows pair; 2048 / 4096 rows 1 / 2.5 % faster).
bool gemm_tc_swiglu_supported(int F, int K, int B) {
  return F >= 1 && K >= kBK && K % kBK == 0 && B >= 1024 && B <= 65535 * kSwBN;
}

cudaError_t launch_gemm_tc_swiglu(const void* W, const void* X, int F, int K, int B, void* h, const Launch& L) {
  if (!gemm_tc_swiglu_supported(F, K, B)) return cudaErrorInvalidValue;
  CUtensorMap tw, tx;
  cudaError_t e = encode_rowmajor_bf16(&tw, W, (uint64_t)2 * F, (uint64_t)K, kBM);
  if (e != cudaSuccess) return e;
  e = encode_rowmajor_bf16(&tx, X, (uint64_t)B, (uint64_t)K, kSwBN);
  if (e != cudaSuccess) return e;
  if (gemm_wide_persistent()) {
    // persistent form: 64 gate rows over 64 up rows per weight tile (two 64-row boxes)
    e = encode_rowmajor_bf16(&tw, W, (uint64_t)2 * F, (uint64_t)K, kBM / 2);
    if (e != cudaSuccess) return e;
    TcParams tp = {};
    tp.R = 2 * F; tp.K = K; tp.B = B; tp.err = L.err;
    const int items = ceil_div(F, kBM / 2) * ceil_div(B, kWdBN);
    const int grid = std::min(items, dev_info().sm_count);
    static bool wd_attr_set = false;
    if (!wd_attr_set) {
      e = cudaFuncSetAttribute(gemm_wide_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wd_smem(true));
      if (e != cudaSuccess) return e;
      wd_attr_set = true;
    }
    return launch_ex(gemm_wide_kernel<true>, dim3(grid), dim3(kWdThreads), wd_smem(true), L, tw, tx, tp,
                     (__nv_bfloat16*)h, F);
  }
  SwParams p = {};
  p.F = F; p.K = K; p.B = B; p.h = (__nv_bfloat16*)h; p.err = L.err;
  const size_t smem = 1024 + (size_t)kSwSt * (2 * kTileA + kTileX256) + (2 * kSwSt + 1) * 8 + 16;
  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(gemm_tc_swiglu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(gemm_tc_swiglu_kernel, dim3(ceil_div(B, kSwBN), ceil_div(F, kBM)), dim3(kThreadsTc), smem, L, tw,
                   tx, p);
}

}  // namespace qd
