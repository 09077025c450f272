// W4A16 weight-streaming GEMV (batch 1) on the tcgen05 tensor cores.
//
// "GPU Kernel Lab" README, "Quantization experiments" and "qwen3-8b-rtx4080-cutedsl"
// README, "W4A16 dequant-fused GEMM": INT4 weights with one scale per output row,
// dequantised inside the weight stream. Same format and results as gemv_w4.cu
// (codes q = u - 8 as offset-binary nibbles, the even column low; w = f32(d) q).
//
// An alternative to the mma.sync form (selected by QD_W4_IMPL=tc). The products run
// on tcgen05 and the SM only converts; measured, it is slower: the conversion (about
// 0.9 ALU instruction per weight) alone streams 3.35 TB/s of codes on the LM head,
// the weight boxes alone 6.07 TB/s, and the MMA handshakes add to the conversion
// instead of hiding under it (the whole kernel 2.3 TB/s against 3.0 for mma.sync).
//   * A = the weight rows, converted to exact bf16 codes in TMEM: a 128-row tile
//     is one row per TMEM lane; 8 converter warps read the rows of each staged
//     tile (TMA, 128-byte swizzle: a thread reading its own row hits distinct
//     banks) and write bf16 code pairs with tcgen05.st. Each 32-bit word of 8
//     nibbles gives four pairs (nibbles j and j + 4): (w >> 4j) & 0x000F000F |
//     0x43004300 is 128 + u in bf16, and one bf16x2 subtraction of 136 gives q.
//   * B = the activation, staged once in shared memory in the same pair order
//     (x[8G + j], x[8G + j + 4]). Its K-major descriptor steps 16 bytes between
//     core matrices along K and the 8 rows of a core matrix are 16 bytes apart, so
//     column n of B reads x shifted by 8n elements: column 0 is x itself, the
//     other columns are ignored. B costs the activation's own 2 bytes per column.
//   * D = 128 x 16 f32 in TMEM (M = 128, N = 16, K = 16 per instruction); column 0
//     of each lane is the row's sum q x, exact products in f32 accumulation.
// The work is (128-row tile, K range) items: tiles whose count underfills the SMs
// split K, and the tile's last split (ticket) adds the partials in split order.
// Warp roles: 0 producer (TMA), 1 MMA issuer, 2..9 converters, 10..13 epilogue;
// every wait is bounded. Epilogues: store, residual add, paired gate/up SwiGLU,
// and the LM head's local top-k with a ticketed merge and the state advance.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <cuda.h>

#include <algorithm>
#include <climits>
#include <cstdlib>

namespace qd {
namespace {

constexpr int kTR = 128;                 // weight rows per tile (MMA M, TMEM lanes)
constexpr int kKB = 256;                 // K per staged box (128 bytes of codes per row)
constexpr int kBoxBytes = kTR * kKB / 2; // 16 KB
constexpr int kNS = 8;                   // staged boxes in the ring
constexpr int kNA = 3;                   // TMEM A buffers (128 columns each)
constexpr int kDCols = 32;               // per D buffer: gate (0..15) and up (16..31)
constexpr int kAcol0 = 2 * kDCols;       // first A column
constexpr int kTmemCols = 512;
constexpr int kConvWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kWarpsTc = 2 + kConvWarps + kEpiWarps;
constexpr int kThreadsW4 = 32 * kWarpsTc;       // 448
constexpr int kWorkThreads = kThreadsW4 - 32;    // every warp but the producer
constexpr int kMaxK = 16384;
constexpr int kMaxG = kMaxK / 8 / kWorkThreads + 1;   // 8-column activation groups per thread
constexpr int kMaxTopK = 16;
constexpr int kMaxKeep = 2560;           // rows one CTA keeps for the top-k (and the merge's candidates)

struct W4TcParams {
  int R, K, n_kb;              // n_kb = K / 256
  int pair, pair_F;            // EPI_SWIGLU: tiles of gate rows, up rows at + pair_F
  int n_tiles, splits, n_items;
  const __half* d;
  int pro;
  const void* x;
  const __nv_bfloat16* norm_w;
  float eps;
  int epi;
  float* y;
  __nv_bfloat16* y_bf16;
  float* part;                 // splits > 1: [tiles][splits][2][128] partial sums
  int* cnt;                    // [tiles] tickets, zero between launches
  int* err;
  int trig_late;
  int w_evict_first;
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

// ---- tcgen05 wrappers
QD_DEV void t_alloc(uint32_t* slot) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(kTmemCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
QD_DEV void t_dealloc(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kTmemCols) : "memory");
}
QD_DEV void t_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
QD_DEV void t_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
QD_DEV void t_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// D (f32) += A (bf16, TMEM) . B (bf16, shared memory), M = 128, N = 16, K = 16
constexpr uint32_t kIdescW4 = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(16 >> 3) << 17) |
                              ((uint32_t)(kTR >> 4) << 24);
QD_DEV void t_mma(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(kIdescW4), "r"(accumulate)
      : "memory");
}
// B descriptor: K-major, no swizzle; 16 bytes between core matrices along K (the
// leading offset) and 128 between 8-row groups (the stride offset)
QD_DEV uint64_t b_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)(16 >> 4) << 16;
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}
// 64 columns of 32 bits into this warp's 32 TMEM lanes
QD_DEV void t_st64(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
      "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
      "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]),
      "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]),
      "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]),
      "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]),
      "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
      : "memory");
}
QD_DEV void t_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// one 32-bit column of this warp's 32 lanes
QD_DEV float t_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  return __uint_as_float(r);
}

QD_DEV uint32_t code_pair(uint32_t w, int j) {   // nibbles (j, j + 4) -> bf16 (q_j, q_j+4)
  const uint32_t v = ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x43084308u));   // 0x4308: bf16 136
  return r;
}
QD_DEV uint32_t bf16_bits_w4(float f) { return __float_as_uint(f) >> 16; }   // f already a bf16 value
QD_DEV float silu_w4(float g) { return g / (1.0f + expf(-g)); }

struct CandW4 {
  float v;
  int i;
};
QD_DEV bool better_w4(const CandW4& a, const CandW4& b) { return a.v > b.v || (a.v == b.v && a.i < b.i); }

// named barrier among the 128 epilogue threads
QD_DEV void epi_sync() { asm volatile("bar.sync 2, %0;" ::"n"(32 * kEpiWarps) : "memory"); }
// named barrier among every thread but the producer warp
QD_DEV void work_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kWorkThreads) : "memory"); }

// best candidate among the epilogue threads; sh: [kEpiWarps] scratch
QD_DEV CandW4 epi_best(CandW4 c, CandW4* sh) {
  const int lane = threadIdx.x & 31, ew = (threadIdx.x >> 5) - (2 + kConvWarps);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    CandW4 d;
    d.v = __shfl_xor_sync(0xffffffffu, c.v, o);
    d.i = __shfl_xor_sync(0xffffffffu, c.i, o);
    if (better_w4(d, c)) c = d;
  }
  if (lane == 0) sh[ew] = c;
  epi_sync();
  CandW4 b = sh[0];
#pragma unroll
  for (int w = 1; w < kEpiWarps; ++w)
    if (better_w4(sh[w], b)) b = sh[w];
  epi_sync();
  return b;
}

__global__ void __launch_bounds__(kThreadsW4, 1)
    gemv_w4_tc_kernel(const __grid_constant__ CUtensorMap tmW, const W4TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* ring = smem;                                        // [kNS][128 rows x 128 B]
  unsigned char* xs = ring + (size_t)kNS * kBoxBytes;                // activation pairs [K] + 256 B
  uint64_t* bars = (uint64_t*)(xs + (size_t)p.K * 2 + 256);
  uint64_t* full = bars;                 // [kNS] box landed
  uint64_t* empty = full + kNS;          // [kNS] box read by its 4 converter warps
  uint64_t* afull = empty + kNS;         // [kNA] A buffer written (its 4 converter warps)
  uint64_t* aempty = afull + kNA;        // [kNA] A buffer read by the MMAs (commit)
  uint64_t* dfull = aempty + kNA;        // [2] D complete (commit)
  uint64_t* dempty = dfull + 2;          // [2] D read by the 4 epilogue warps
  uint32_t* tmem_slot = (uint32_t*)(dempty + 2);
  float* keep_v = (float*)(tmem_slot + 4);     // EPI_TOPK: [kMaxKeep] values, then rows
  int* keep_i = (int*)(keep_v + kMaxKeep);
  __shared__ float s_ss[kWarpsTc];
  __shared__ CandW4 s_c[kEpiWarps];
  __shared__ int s_last, s_ticket;
  __shared__ int s_got[kEpiWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x;
  const int n_my = p.n_items > (int)blockIdx.x ? (p.n_items - 1 - (int)blockIdx.x) / G + 1 : 0;
  const int tiles_per = p.pair ? 2 : 1;

  if (tid == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConvWarps / 2);   // the 4 warps of one parity
    }
    for (int i = 0; i < kNA; ++i) {
      mbar_init(&afull[i], kConvWarps / 2);
      mbar_init(&aempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&dfull[i], 1);
      mbar_init(&dempty[i], kEpiWarps);
    }
    fence_mbar_init();
  }
  if (warp == 1) t_alloc(tmem_slot);
  t_fence_before();
  __syncthreads();
  t_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (!p.trig_late) pdl_launch_dependents();

  // the K blocks [kb0, kb1) and tile of this CTA's item number `it`
  auto item_of = [&](int it, int& tile, int& split, int& kb0, int& kb1) {
    const int item = (int)blockIdx.x + it * G;
    tile = item / p.splits;
    split = item - tile * p.splits;
    kb0 = (int)(((long long)p.n_kb * split) / p.splits);
    kb1 = (int)(((long long)p.n_kb * (split + 1)) / p.splits);
  };

  if (warp == 0) {
    // ---- producer: weights only, so no dependency wait; as far ahead as the ring allows
    if (lane == 0) {
      int sc = 0;
      bool ok = true;
      for (int it = 0; it < n_my && ok; ++it) {
        int tile, split, kb0, kb1;
        item_of(it, tile, split, kb0, kb1);
        for (int kb = kb0; kb < kb1 && ok; ++kb)
          for (int t = 0; t < tiles_per; ++t, ++sc) {
            const int slot = sc % kNS;
            if (sc >= kNS && !mbar_wait_bounded(&empty[slot], (uint32_t)(((sc / kNS) - 1) & 1), p.err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[slot], kBoxBytes);
            const int row = (t ? p.pair_F : 0) + tile * kTR;
            tma_load_2d(ring + (size_t)slot * kBoxBytes, &tmW, kb * (kKB / 2), row, &full[slot]);
          }
      }
      // every copy issued has landed before this CTA may exit
      for (int i = max(0, sc - kNS); i < sc; ++i)
        mbar_wait_bounded(&full[i % kNS], (uint32_t)((i / kNS) & 1), p.err);
    }
    __syncwarp();
  } else {
    // ---- the activation, once, as bf16 pairs (x[8G + j], x[8G + j + 4]) for j < 4,
    // plus 256 zero bytes read past the end by the shifted B columns
    const int wt = tid - 32;
    const int NGK = p.K / 8;
    uint4 wn[kMaxG];
#pragma unroll
    for (int j = 0; j < kMaxG; ++j) {
      const int g8 = wt + j * kWorkThreads;
      wn[j] = (p.pro == PRO_RMSNORM && g8 < NGK) ? *(const uint4*)(p.norm_w + 8 * g8) : make_uint4(0u, 0u, 0u, 0u);
    }
    pdl_wait();
    float xv[kMaxG][8];
#pragma unroll
    for (int j = 0; j < kMaxG; ++j) {
      const int g8 = wt + j * kWorkThreads;
#pragma unroll
      for (int e = 0; e < 8; ++e) xv[j][e] = 0.f;
      if (g8 >= NGK) continue;
      if (p.pro == PRO_X_BF16) {
        const uint4 v = *(const uint4*)((const __nv_bfloat16*)p.x + 8 * g8);
        xv[j][0] = bf_lo(v.x); xv[j][1] = bf_hi(v.x); xv[j][2] = bf_lo(v.y); xv[j][3] = bf_hi(v.y);
        xv[j][4] = bf_lo(v.z); xv[j][5] = bf_hi(v.z); xv[j][6] = bf_lo(v.w); xv[j][7] = bf_hi(v.w);
      } else {
        const float4 a = *(const float4*)((const float*)p.x + 8 * g8);
        const float4 b = *(const float4*)((const float*)p.x + 8 * g8 + 4);
        xv[j][0] = a.x; xv[j][1] = a.y; xv[j][2] = a.z; xv[j][3] = a.w;
        xv[j][4] = b.x; xv[j][5] = b.y; xv[j][6] = b.z; xv[j][7] = b.w;
      }
    }
    if (p.pro == PRO_X_F32) {
#pragma unroll
      for (int j = 0; j < kMaxG; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[j][e] = round_bf16(xv[j][e]);
    } else if (p.pro == PRO_RMSNORM) {
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxG; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(xv[j][e], xv[j][e], ss);
      ss = warp_sum(ss);
      if (lane == 0) s_ss[warp] = ss;
      work_sync();
      float tot = 0.f;
      for (int w = 1; w < kWarpsTc; ++w) tot += s_ss[w];
      const float inv = 1.0f / sqrtf(tot / (float)p.K + p.eps);
#pragma unroll
      for (int j = 0; j < kMaxG; ++j) {
        const uint4 w = wn[j];
        const float nw[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y),
                             bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[j][e] = round_bf16(nw[e] * round_bf16(xv[j][e] * inv));
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxG; ++j) {
      const int g8 = wt + j * kWorkThreads;
      if (g8 >= NGK + 16) continue;       // the activation, then 256 zero bytes
      uint4 v;
      v.x = bf16_bits_w4(xv[j][0]) | (bf16_bits_w4(xv[j][4]) << 16);
      v.y = bf16_bits_w4(xv[j][1]) | (bf16_bits_w4(xv[j][5]) << 16);
      v.z = bf16_bits_w4(xv[j][2]) | (bf16_bits_w4(xv[j][6]) << 16);
      v.w = bf16_bits_w4(xv[j][3]) | (bf16_bits_w4(xv[j][7]) << 16);
      *(uint4*)(xs + (size_t)16 * g8) = v;
    }
    fence_proxy_async_smem();   // the tensor cores read these stores through the async proxy
    work_sync();

    if (warp == 1) {
      // ---- MMA issuer: D[dbuf] (+16 for the up tile) = sum over K of A . B
      if (lane == 0) {
        const uint32_t xs_u = smem_u32(xs);
        int sc = 0;
        bool ok = true;
        for (int it = 0; it < n_my && ok; ++it) {
          int tile, split, kb0, kb1;
          item_of(it, tile, split, kb0, kb1);
          const int dbuf = it & 1;
          if (it >= 2 && !mbar_wait_bounded(&dempty[dbuf], (uint32_t)(((it >> 1) - 1) & 1), p.err)) {
            break;
          }
          t_fence_after();
          for (int kb = kb0; kb < kb1 && ok; ++kb)
            for (int t = 0; t < tiles_per; ++t, ++sc) {
              const int buf = sc % kNA;
              if (!mbar_wait_bounded(&afull[buf], (uint32_t)((sc / kNA) & 1), p.err)) {
                ok = false;
                break;
              }
              t_fence_after();
              const uint32_t d_t = tmem + (uint32_t)(dbuf * kDCols + t * 16);
              const uint32_t a_t = tmem + (uint32_t)(kAcol0 + buf * 128);
#pragma unroll
              for (int i = 0; i < kKB / 16; ++i)
                t_mma(d_t, a_t + (uint32_t)(8 * i), b_desc(xs_u + (uint32_t)(2 * (kb * kKB + 16 * i))),
                      (kb != kb0 || i > 0) ? 1u : 0u);
              t_commit(&aempty[buf]);   // the A buffer is free once these MMAs have read it
            }
          if (ok) t_commit(&dfull[dbuf]);
        }
        // nothing of this thread's is still running on the tensor cores past here
        if (sc > 0) mbar_wait_bounded(&aempty[(sc - 1) % kNA], (uint32_t)(((sc - 1) / kNA) & 1), p.err);
      }
      __syncwarp();
    }

    if (warp >= 2 && warp < 2 + kConvWarps) {
      // ---- converters: warp (quarter q, parity h) takes TMEM lanes 32q .. 32q + 31 (its
      // tile rows) of every staged box with sc % 2 == h, so two boxes are converted at
      // once; a thread converts its row's 32 words (128 bf16 code pairs)
      const int q = warp & 3, h = (warp - 2) >> 2;
      const int row = 32 * q + lane;
      int sc = 0;
      bool ok = true;
      for (int it = 0; it < n_my && ok; ++it) {
        int tile, split, kb0, kb1;
        item_of(it, tile, split, kb0, kb1);
        for (int kb = kb0; kb < kb1 && ok; ++kb)
          for (int t = 0; t < tiles_per; ++t, ++sc) {
            if ((sc & 1) != h) continue;
            const int slot = sc % kNS, buf = sc % kNA;
            if (!mbar_wait_bounded(&full[slot], (uint32_t)((sc / kNS) & 1), p.err)) {
              ok = false;
              break;
            }
            const unsigned char* rb = ring + (size_t)slot * kBoxBytes + (size_t)row * 128;
            uint4 v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) v[c] = *(const uint4*)(rb + ((c ^ (row & 7)) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (sc >= kNA && !mbar_wait_bounded(&aempty[buf], (uint32_t)(((sc / kNA) - 1) & 1), p.err)) {
              ok = false;
              break;
            }
            t_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint32_t r[64];
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const uint4 vv = v[4 * half + c];
                const uint32_t wv[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                  for (int j = 0; j < 4; ++j) r[4 * (4 * c + e) + j] = code_pair(wv[e], j);
              }
              t_st64(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kAcol0 + buf * 128 + 64 * half), r);
            }
            t_wait_st();
            t_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[buf]);
          }
      }
    } else if (warp >= 2 + kConvWarps) {
      // ---- epilogue: lane quarter q, tile row 32q + lane
      const int q = warp & 3;
      const int rit = 32 * q + lane;
      const bool topk = p.epi == EPI_TOPK;
      bool epi_failed = false;
      auto finish = [&](int it, int tile, float g, float u) {
        if (p.pair) {
          const int j = tile * kTR + rit;
          if (j < p.pair_F) {
            const float gv = __half2float(p.d[j]) * g;
            const float uv = __half2float(p.d[p.pair_F + j]) * u;
            p.y_bf16[j] = __float2bfloat16_rn(silu_w4(gv) * uv);
          }
          return;
        }
        const int r = tile * kTR + rit;
        float v = __int_as_float(0x7fffffff);
        if (r < p.R) {
          v = __half2float(p.d[r]) * g;
          if (p.epi == EPI_RESID_ADD) p.y[r] += v;
          else p.y[r] = v;
        }
        if (topk) {
          keep_v[it * kTR + rit] = v;   // NaN past the last row: never chosen
          keep_i[it * kTR + rit] = r;
        }
      };
      for (int it = 0; it < n_my; ++it) {
        int tile, split, kb0, kb1;
        item_of(it, tile, split, kb0, kb1);
        const int dbuf = it & 1;
        const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(&dfull[dbuf], (uint32_t)((it >> 1) & 1), p.err));
        if (lane == 0) s_got[warp - 2 - kConvWarps] = got;
        epi_sync();   // the four epilogue warps take the same decision
        if (!(s_got[0] && s_got[1] && s_got[2] && s_got[3])) {
          epi_failed = true;
          break;
        }
        t_fence_after();
        const uint32_t dt = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(dbuf * kDCols);
        const float g = t_ld1(dt);
        const float u = p.pair ? t_ld1(dt + 16) : 0.f;
        t_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[dbuf]);
        if (p.splits == 1) {
          finish(it, tile, g, u);
          continue;
        }
        // publish this split's partials, take the tile's ticket; the last split adds
        // every split's partials in split order
        float* pt = p.part + ((size_t)tile * p.splits + split) * 2 * kTR;
        pt[rit] = g;
        pt[kTR + rit] = u;
        epi_sync();
        if (rit == 0) {
          __threadfence();
          s_last = atomicAdd(p.cnt + tile, 1) == p.splits - 1;
        }
        epi_sync();
        if (s_last) {
          __threadfence();
          const float* pb = p.part + (size_t)tile * p.splits * 2 * kTR;
          float gs = 0.f, us = 0.f;
          for (int sp = 0; sp < p.splits; ++sp) {
            gs += __ldcg(pb + (size_t)sp * 2 * kTR + rit);
            us += __ldcg(pb + (size_t)sp * 2 * kTR + kTR + rit);
          }
          finish(it, tile, gs, us);
          if (rit == 0) p.cnt[tile] = 0;
        }
        epi_sync();
      }
      if (topk && !epi_failed) {
        // ---- this CTA's top k of its rows, then the ticket; the last CTA merges
        const int k = p.top_k, nk = n_my * kTR;
        epi_sync();
        for (int sel = 0; sel < k; ++sel) {
          CandW4 c = {-INFINITY, INT_MAX};
          for (int e = rit; e < nk; e += kTR) {
            const float v = keep_v[e];
            if (isnan(v)) continue;
            const CandW4 d = {v, keep_i[e]};
            if (better_w4(d, c)) c = d;
          }
          c = epi_best(c, s_c);
          for (int e = rit; e < nk; e += kTR)
            if (c.i != INT_MAX && keep_i[e] == c.i) keep_v[e] = __int_as_float(0x7fffffff);   // taken
          if (rit == 0) {
            p.cand_v[(size_t)blockIdx.x * k + sel] = c.v;
            p.cand_i[(size_t)blockIdx.x * k + sel] = c.i;
          }
          epi_sync();
        }
        if (rit == 0) {
          __threadfence();
          s_ticket = atomicAdd(p.ticket, 1);
        }
        epi_sync();
        if (s_ticket == G - 1) {
          __threadfence();
          const int nc = G * k;
          for (int e = rit; e < nc; e += kTR) {
            keep_v[e] = __ldcg(p.cand_v + e);
            keep_i[e] = __ldcg(p.cand_i + e);
          }
          epi_sync();
          int first = INT_MAX;
          for (int sel = 0; sel < k; ++sel) {
            CandW4 c = {-INFINITY, INT_MAX};
            for (int e = rit; e < nc; e += kTR) {
              const CandW4 d = {keep_v[e], keep_i[e]};
              if (!isnan(d.v) && d.i != INT_MAX && better_w4(d, c)) c = d;
            }
            c = epi_best(c, s_c);   // every row is a candidate of one CTA at most
            for (int e = rit; e < nc; e += kTR)
              if (c.i != INT_MAX && keep_i[e] == c.i) keep_v[e] = __int_as_float(0x7fffffff);
            if (rit == 0) {
              if (p.topk_ids) p.topk_ids[sel] = c.i == INT_MAX ? -1 : c.i;
              if (p.topk_vals) p.topk_vals[sel] = c.v;
              if (sel == 0) first = c.i;
            }
            epi_sync();
          }
          if (rit == 0) {
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
      }
    }
  }
  pdl_launch_dependents();
  t_fence_before();
  __syncthreads();
  t_fence_after();
  if (warp == 1) t_dealloc(tmem);
}

}  // namespace

// ---------------------------------------------------------------- host
namespace {

constexpr int kMaxSplitTilesW4 = 4096;      // ticket block at the start of the workspace

int w4_tiles(int R, bool pair) { return ceil_div(pair ? R / 2 : R, kTR); }

// K splits: tiles that underfill the SMs split K so that about one item per SM
// streams (at least one 256-column block each)
int w4_splits(int R, int K, bool pair) {
  const int tiles = w4_tiles(R, pair), n_kb = K / kKB, sms = dev_info().sm_count;
  if (tiles >= sms || tiles > kMaxSplitTilesW4) return 1;
  return std::max(1, std::min(n_kb, ceil_div(sms, tiles)));
}

size_t smem_w4_tc(int K, bool topk) {
  return 1024 + (size_t)kNS * kBoxBytes + (size_t)K * 2 + 256 + (2 * kNS + 2 * kNA + 4) * 8 + 16 +
         (topk ? (size_t)kMaxKeep * 8 : 0);
}

}  // namespace

// QD_W4_IMPL (read on every call): "tc" runs the GEMVs whose K is a multiple of 256
// on this form; anything else keeps the mma.sync form (gemv_w4.cu), measured faster.
bool gemv_w4_tc_supported(int K) {
  const char* v = getenv("QD_W4_IMPL");
  const bool on = v && v[0] == 't' && v[1] == 'c';
  return on && K >= kKB && K % kKB == 0 && K <= kMaxK;
}

size_t gemv_w4_tc_workspace_bytes(int R, int K, bool pair) {
  if (K < kKB || K % kKB) return 0;
  const int sp = w4_splits(R, K, pair);
  if (sp <= 1) return 0;
  return (size_t)kMaxSplitTilesW4 * 4 + (size_t)w4_tiles(R, pair) * sp * 2 * kTR * 4;
}

cudaError_t launch_gemv_w4_tc(const GemvW4Args& a, void* ws, size_t ws_bytes, const Launch& L) {
  if (!gemv_w4_tc_supported(a.K) || a.R < 1) return cudaErrorInvalidValue;
  const bool pair = a.epi == EPI_SWIGLU, topk = a.epi == EPI_TOPK;
  if (pair && a.R % 2) return cudaErrorInvalidValue;
  if (topk && (a.top_k < 1 || a.top_k > kMaxTopK || !a.ws)) return cudaErrorInvalidValue;
  CUtensorMap tm;
  cudaError_t e = encode_tmap_u8_sw128(&tm, a.W, (uint64_t)a.R, (uint64_t)a.K / 2, kTR);
  if (e != cudaSuccess) return e;
  W4TcParams p = {};
  p.R = a.R; p.K = a.K; p.n_kb = a.K / kKB;
  p.pair = pair ? 1 : 0; p.pair_F = pair ? a.R / 2 : 0;
  p.n_tiles = w4_tiles(a.R, pair);
  p.splits = 1;
  const size_t need = gemv_w4_tc_workspace_bytes(a.R, a.K, pair);
  if (!topk && ws && need > 0 && ws_bytes >= need) {
    p.splits = w4_splits(a.R, a.K, pair);
    p.cnt = (int*)ws;
    p.part = (float*)((unsigned char*)ws + (size_t)kMaxSplitTilesW4 * 4);
  }
  p.n_items = p.n_tiles * p.splits;
  const int grid = std::max(1, std::min(p.n_items, dev_info().sm_count));
  if (topk && ceil_div(p.n_items, grid) * kTR > kMaxKeep) return cudaErrorInvalidValue;
  if (topk && grid * a.top_k > kMaxKeep) return cudaErrorInvalidValue;
  p.d = (const __half*)a.d;
  p.pro = a.pro; p.x = a.x; p.norm_w = (const __nv_bfloat16*)a.norm_w; p.eps = a.eps;
  p.epi = a.epi; p.y = a.y; p.y_bf16 = (__nv_bfloat16*)a.y_bf16;
  p.err = L.err; p.trig_late = L.trig_late; p.w_evict_first = a.w_evict_first;
  if (topk) {
    unsigned char* tw = (unsigned char*)a.ws;
    const size_t cb = (((size_t)dev_info().sm_count * kMaxTopK * 8 + 255) & ~(size_t)255);
    p.top_k = a.top_k;
    p.cand_v = (float*)tw;
    p.cand_i = (int*)(tw + (size_t)dev_info().sm_count * kMaxTopK * 4);
    p.ticket = (int*)(tw + cb);
    p.tok = a.tok; p.pos = a.pos; p.step = a.step; p.out_tokens = a.out_tokens; p.max_steps = a.max_steps;
    p.topk_ids = a.topk_ids; p.topk_vals = a.topk_vals;
  }
  const size_t smem = smem_w4_tc(a.K, topk);
  if (smem > (size_t)dev_info().max_smem_optin) return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(gemv_w4_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_w4_tc(kMaxK, true));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(gemv_w4_tc_kernel, dim3(grid), dim3(kThreadsW4), smem, L, tm, p);
}

}  // namespace qd
