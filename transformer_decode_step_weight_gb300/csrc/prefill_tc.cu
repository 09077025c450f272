// Causal prefill attention on the tcgen05 tensor cores.
//
// "qwen3-8b-rtx4080-cutedsl" README, "Flash Attention 2": the prompt's rows attend
// causally in key tiles with an online softmax, the score and probability tiles never
// leaving the chip; "GQA + QK-Norm": per-head RMSNorm of q and RoPE before the scores.
// Row i of the prompt sits at position pos[0] + i and attends to keys 0 .. pos[0] + i.
//
// GB300 layout: one CTA per (128 query rows, q head). The queries (norm, RoPE, softmax
// scale with log2 e folded in) are staged once as bf16 hi + lo in 128-byte-swizzled
// K-major tiles. Per 64-key tile:
//   * S[128 x 64] = Q K^T on tcgen05 into TMEM (16 MMAs: M 128, N 64, K 16, the hi and
//     the lo half of q), K streamed by TMA from a packed copy of the kv head's keys;
//   * the threads of each query row (its TMEM lane) load its 64 scores, mask keys past
//     its position, and keep a reference maximum that moves only when
//     a score passes it by more than 8 (a factor 256) so the accumulator in TMEM is
//     rescaled rarely; p = exp2(s - m_ref) goes to shared memory as bf16 hi + lo in
//     the swizzled layout the MMA reads;
//   * O[128 x 128] += P V on tcgen05 (8 MMAs: M 128, N 128, K 16) with V streamed as a
//     transposed copy [128 dims x keys], so both operands are K-major.
// Producer threads keep two K and two V tiles in flight, refilling a stage as soon as its
// MMAs are done, and an issuer thread issues S of the next tiles while the rows finish
// the current one. Every wait is bounded.
// Each query row is shared by two threads in two warps (TMEM lane quarters are per warp
// modulo 4), each taking half of the tile's keys, so two row warps run per SM sub-partition.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_common.cuh"

#include <cuda.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>

namespace qd {
namespace {

constexpr int kD = 128;
constexpr int kQT = 128;               // query rows per CTA (the MMA's M, TMEM lanes)
constexpr int kKT = 64;                // keys per tile (S columns)
constexpr int kKSt = 3;                // K ring stages
constexpr int kVSt = 2;                // V^T ring stages
constexpr int kQChunk = kQT * 128;     // [128 rows x 64 bf16] swizzled chunk: 16 KB
constexpr int kKChunk = kKT * 128;     // [64 keys x 64 bf16]: 8 KB
constexpr int kKTile = 2 * kKChunk;    // a K tile: dims 0-63, 64-127
constexpr int kVTile = kD * 128;       // a V^T tile [128 dims x 64 keys]: 16 KB
constexpr int kRowWarps = 8;           // two warps per TMEM lane quarter (32 of a tile's 64 keys each)
constexpr int kIssuer = kRowWarps;     // the MMA issuer warp
constexpr int kProdK = kRowWarps + 1;  // the K producer warp
constexpr int kProdV = kRowWarps + 2;  // the V^T producer warp
constexpr int kThreads = 32 * (kRowWarps + 3);
constexpr int kOffQh = 0;
constexpr int kOffQl = kOffQh + 2 * kQChunk;
constexpr int kOffK = kOffQl + 2 * kQChunk;      // K ring [kKSt]
constexpr int kOffV = kOffK + kKSt * kKTile;     // V^T ring [kVSt]
constexpr int kOffPh = kOffV + kVSt * kVTile;    // P hi [2 buffers]
constexpr int kOffPl = kOffPh + 2 * kQChunk;     // P lo [2 buffers]
constexpr int kOffBar = kOffPl + 2 * kQChunk;
constexpr int kOffXm = kOffBar + 256;            // the row pairs' traded maxima / sums [2][2][kQT] f32
constexpr size_t kSmem = (size_t)kOffXm + 2 * 2 * kQT * 4 + 1024;   // slack for the 1024-byte alignment
constexpr int kSBuf = 3;               // TMEM S buffers: S of tile i + 3 goes out behind P V of tile i
constexpr uint32_t kTmemCols = 512;    // S buffers at columns 0, 64, 128; O at column 256 (128)
constexpr uint32_t kTmemO = 256;
constexpr float kRescale = 8.0f;       // log2 units a score may pass the reference maximum

struct TcPfParams {
  const float* qkv;                    // f32 [n, (Hq + 2 Hkv) D]
  int n, Hq, Hkv;
  const __nv_bfloat16* q_norm;
  const float2* rope;
  int rope_max_pos;
  float eps;
  int act_bf16;
  const int32_t* pos;                  // pos[0]: the first prompt row's position
  int L;                               // keys per kv head in the packed copies (a multiple of 64)
  int cap;                             // cache capacity in tokens
  float scale_log2;
  __nv_bfloat16* out;                  // bf16 [n, Hq D]
  int* err;
};

QD_DEV uint32_t pack_bf(float lo, float hi) { return f2bf_bits(lo) | (f2bf_bits(hi) << 16); }
// bf16(lo) in the low half, bf16(hi) in the high half, both rounded to nearest even by
// one paired conversion
QD_DEV uint32_t bf2_bits(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  uint32_t u;
  memcpy(&u, &v, 4);
  return u;
}
// 2^x by the hardware's approximate base-2 exponential (-inf gives +0, subnormal
// results flush to zero); the relative error is far below the bf16 hi + lo weights'
QD_DEV float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                           const TcPfParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bar = (uint64_t*)(smem + kOffBar);
  uint64_t* k_full = bar;         // [kKSt] a K tile landed
  uint64_t* k_empty = bar + 3;    // [kKSt] its S MMAs are done with it
  uint64_t* v_full = bar + 6;     // [kVSt] a V^T tile landed
  uint64_t* v_empty = bar + 8;    // [kVSt] its P V MMAs are done with it (and with that P buffer)
  uint64_t* s_full = bar + 10;    // [kSBuf] S of a tile in its TMEM buffer
  uint64_t* p_full = bar + 13;    // [2] 128 rows read S and wrote P into that buffer (O rescaled)
  uint64_t* o_done = bar + 15;    // [2] the P V MMAs of a tile completed
  uint64_t* x_bar = bar + 17;     // [2 parities][4 lane quarters] both warps of a pair traded (64 lanes)
  uint32_t* tslot = (uint32_t*)(bar + 25);
  int* s_abort = (int*)(tslot + 1);
  float* xm = (float*)(smem + kOffXm);

  // grid (q head, query tile), blocks dispatched in that order: the longest query tiles
  // of every head first, so the short ones fill the SMs at the end of the causal
  // triangle (head by head, the last heads' longest tiles would start late and run alone)
  const int h = blockIdx.x, qt = (int)(gridDim.y - 1 - blockIdx.y);
  const int g = h / (p.Hq / p.Hkv);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  pdl_wait();   // q, the packed K / V come from the kernels before this one
  pdl_launch_dependents();
  const int pos0 = p.pos[0];
  if (pos0 < 0 || pos0 + p.n > p.cap || pos0 + p.n > p.rope_max_pos || pos0 + p.n > p.L) {
    if (qt == 0 && h == 0 && tid == 0) set_error(p.err, QD_DEVERR_POS);
    return;
  }
  const int r0 = qt * kQT;
  const int nrows = min(kQT, p.n - r0);
  const int kend = pos0 + r0 + nrows;                 // keys [0, kend) are visible to some row
  const int n_kt = (kend + kKT - 1) / kKT;

  if (tid == 0) {
    for (int i = 0; i < kKSt; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < kSBuf; ++i) mbar_init(&s_full[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&p_full[i], kQT * kRowWarps / 4);
      mbar_init(&o_done[i], 1);
    }
    for (int i = 0; i < 8; ++i) mbar_init(&x_bar[i], 64);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, kTmemCols);

  // ---- queries: warp w builds rows 32w .. 32w + 31, four at a time; lane holds dims
  // 4 lane .. + 3 (the arithmetic and order of the mma.sync prefill kernel)
  if (warp < 4) {
    const int qkv_w = (p.Hq + 2 * p.Hkv) * kD;
    const int d0 = 4 * lane;
    const uint2 wq = *(const uint2*)(p.q_norm + d0);
    const float nw[4] = {bf_lo(wq.x), bf_hi(wq.x), bf_lo(wq.y), bf_hi(wq.y)};
    constexpr int kRB = 4;
    for (int rb = 0; rb < 32; rb += kRB) {
      float4 xr[kRB];
      float4 cr[kRB][2];
#pragma unroll
      for (int i = 0; i < kRB; ++i) {
        const int row = r0 + warp * 32 + rb + i;
        if (row < p.n) {
          xr[i] = *(const float4*)(p.qkv + (size_t)row * qkv_w + (size_t)h * kD + d0);
          const float4* cs = (const float4*)(p.rope + (size_t)(pos0 + row) * (kD / 2) + (d0 & 63));
          cr[i][0] = cs[0];
          cr[i][1] = cs[1];
        } else {
          xr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          cr[i][0] = cr[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int i = 0; i < kRB; ++i) {
        const int lr = warp * 32 + rb + i, row = r0 + lr;
        float qv[4] = {0.f, 0.f, 0.f, 0.f};
        if (row < p.n) {   // uniform over the warp
          const float xs[4] = {xr[i].x, xr[i].y, xr[i].z, xr[i].w};
          const float ss = warp_sum(xs[0] * xs[0] + xs[1] * xs[1] + xs[2] * xs[2] + xs[3] * xs[3]);
          const float inv = 1.0f / sqrtf(ss / (float)kD + p.eps);
          float y[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float nv = xs[e] * inv;
            if (p.act_bf16) nv = round_bf16(nv);
            y[e] = nw[e] * nv;
            if (p.act_bf16) y[e] = round_bf16(y[e]);
          }
          const float cc[4][2] = {{cr[i][0].x, cr[i][0].y}, {cr[i][0].z, cr[i][0].w},
                                  {cr[i][1].x, cr[i][1].y}, {cr[i][1].z, cr[i][1].w}};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float other = __shfl_xor_sync(0xffffffffu, y[e], 16);   // dim d ^ 64
            const float r = lane < 16 ? (y[e] * cc[e][0] - other * cc[e][1]) : (y[e] * cc[e][0] + other * cc[e][1]);
            qv[e] = r * p.scale_log2;
          }
        }
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const __nv_bfloat16 h0 = __float2bfloat16_rn(qv[2 * e]), h1 = __float2bfloat16_rn(qv[2 * e + 1]);
          hi[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
          lo[e] = pack_bf(qv[2 * e] - __bfloat162float(h0), qv[2 * e + 1] - __bfloat162float(h1));
        }
        // dims d0 .. d0 + 3: chunk d0 / 64, 16-byte piece (d0 % 64) / 8, half (d0 % 8) / 4
        const uint32_t o = (uint32_t)((lane >> 4) * kQChunk) + tc::sw128_off(lr, (lane & 15) >> 1) +
                           (uint32_t)((lane & 1) * 8);
        *(uint2*)(smem + kOffQh + o) = make_uint2(hi[0], hi[1]);
        *(uint2*)(smem + kOffQl + o) = make_uint2(lo[0], lo[1]);
      }
    }
    fence_proxy_async_smem();   // the MMAs read these tiles through the async proxy
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tS = tbase, tO = tbase + kTmemO;   // S buffer b at tS + 64 b

  if (warp == kProdK || warp == kProdV) {
    if (lane == 0) {
      // ---- producers: K (or V^T) tile i into stage i % ns as soon as the MMAs of tile
      // i - ns are done with the stage, independent of the issuer's other waits
      const bool is_k = warp == kProdK;
      const int ns = is_k ? kKSt : kVSt;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      int issued = 0;
      for (int i = 0; i < n_kt; ++i) {
        const int st = i % ns;
        if (i >= ns && (!mbar_wait_bounded(&empty[st], (uint32_t)(((i - ns) / ns) & 1), p.err) ||
                        *(volatile int*)s_abort))
          break;
        if (is_k) {
          unsigned char* k = smem + kOffK + st * kKTile;
          mbar_arrive_expect_tx(&full[st], kKTile);
          tma_load_2d(k, &tmK, 0, g * p.L + i * kKT, &full[st]);
          tma_load_2d(k + kKChunk, &tmK, 64, g * p.L + i * kKT, &full[st]);
        } else {
          mbar_arrive_expect_tx(&full[st], kVTile);
          tma_load_2d(smem + kOffV + st * kVTile, &tmV, i * kKT, g * kD, &full[st]);
        }
        issued = i + 1;
      }
      // the last copy into each stage lands before the CTA leaves (bounded; at once when
      // the issuer consumed it). No later phase of the stage's barrier can exist.
      for (int t = issued > ns ? issued - ns : 0; t < issued; ++t)
        mbar_wait_limit(&full[t % ns], (uint32_t)((t / ns) & 1), p.err, 10000000ull);
    }
    __syncwarp();
  } else if (warp == kIssuer) {
    if (lane == 0) {  // ---- MMA issuer
      const uint32_t sQh = smem_u32(smem + kOffQh), sQl = smem_u32(smem + kOffQl);
      const uint32_t sK = smem_u32(smem + kOffK), sV = smem_u32(smem + kOffV);
      const uint32_t sPh = smem_u32(smem + kOffPh), sPl = smem_u32(smem + kOffPl);
      auto mma_s = [&](int i) -> bool {  // S = Q K^T of tile i (K stage i % kKSt) into S buffer i % kSBuf
        const int b = i % kSBuf, kb = i % kKSt;
        if (!mbar_wait_bounded(&k_full[kb], (uint32_t)((i / kKSt) & 1), p.err)) return false;
        tc::fence_after();
        const uint32_t k0 = sK + kb * kKTile, ts = tS + 64 * b;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t qo = (j >> 2) * kQChunk + (j & 3) * 32, ko = (j >> 2) * kKChunk + (j & 3) * 32;
          tc::mma<kKT>(ts, tc::desc_sw128(sQh + qo), tc::desc_sw128(k0 + ko), j != 0);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t qo = (j >> 2) * kQChunk + (j & 3) * 32, ko = (j >> 2) * kKChunk + (j & 3) * 32;
          tc::mma<kKT>(ts, tc::desc_sw128(sQl + qo), tc::desc_sw128(k0 + ko), 1);
        }
        tc::commit(&s_full[b]);
        tc::commit(&k_empty[kb]);
        return true;
      };
      bool ok = true;
      for (int i = 0; i < kSBuf && i < n_kt && ok; ++i) ok = mma_s(i);
      for (int i = 0; i < n_kt && ok; ++i) {
        const int b = i & 1;
        const uint32_t ph = (uint32_t)((i >> 1) & 1);
        // the rows read S(i), wrote P(i) into buffer b and rescaled O where needed
        if (!mbar_wait_bounded(&p_full[b], ph, p.err) || !mbar_wait_bounded(&v_full[b], ph, p.err)) {
          ok = false;
          break;
        }
        tc::fence_after();
        const uint32_t v0 = sV + b * kVTile, p_h = sPh + b * kQChunk, p_l = sPl + b * kQChunk;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma<kD>(tO, tc::desc_sw128(p_h + kk * 32), tc::desc_sw128(v0 + kk * 32), (i | kk) != 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) tc::mma<kD>(tO, tc::desc_sw128(p_l + kk * 32), tc::desc_sw128(v0 + kk * 32), 1);
        tc::commit(&o_done[b]);
        tc::commit(&v_empty[b]);
        // S of tile i + kSBuf into S(i)'s buffer right behind them (the rows read S(i)
        // before they wrote P(i))
        if (i + kSBuf < n_kt && !(ok = mma_s(i + kSBuf))) break;
      }
      if (!ok) *(volatile int*)s_abort = 1;
    }
    __syncwarp();
  } else {
    // ---- query rows: warps w and w + 4 share TMEM lane quarter q = w % 4 (rows 32 q ..
    // 32 q + 31, one per lane); half hf = w / 4 takes key columns 32 hf .. 32 hf + 31 of
    // every tile and O columns 64 hf .. 64 hf + 63. The pair trades its rows' maxima each
    // tile (and the row sums at the end) through shared memory, so both halves move the
    // same reference maximum at the same tile.
    const int q4 = warp & 3, hf = warp >> 2;
    const int r = q4 * 32 + lane, row = r0 + r;
    const bool valid = row < p.n;
    const int rowpos = pos0 + row;
    const uint32_t lanes = (uint32_t)(q4 * 32) << 16;
    float m_ref = -INFINITY, l = 0.f;
    bool fail = false;
    // wait (bounded) on a barrier phase; false in every lane if any lane gave up
    auto wait_all = [&](uint64_t* bb, uint32_t ph) -> bool {
      const bool got = mbar_wait_bounded(bb, ph, p.err) && !*(volatile int*)s_abort;
      return __all_sync(0xffffffffu, got);
    };
    // trade number u with the partner warp: this lane's v in, the partner's value out.
    // A slot is written again two trades later, after the partner has passed the trade
    // in between (and so has read it).
    auto trade = [&](int u, float v, float& other) -> bool {
      const int par = u & 1;
      xm[(par * 2 + hf) * kQT + r] = v;
      mbar_arrive(&x_bar[par * 4 + q4]);
      if (!wait_all(&x_bar[par * 4 + q4], (uint32_t)((u >> 1) & 1))) return false;
      other = xm[(par * 2 + (hf ^ 1)) * kQT + r];
      return true;
    };
    for (int i = 0; i < n_kt; ++i) {
      const int b = i & 1;
      if (!wait_all(&s_full[i % kSBuf], (uint32_t)((i / kSBuf) & 1))) {   // the same decision in every lane
        fail = true;
        break;
      }
      tc::fence_after();
      float s[32];
      tc::ld_32x32(tS + 64 * (i % kSBuf) + lanes + 32 * hf, s);
      const int key0 = i * kKT + 32 * hf;
      // the causal mask (and rows past the prompt) only where these 32 keys cross the
      // diagonal of some row of the warp or the warp holds such rows (warp-uniform)
      const bool masked = key0 + 31 > pos0 + r0 + q4 * 32 || r0 + q4 * 32 + 31 >= p.n;
      if (masked) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (!valid || key0 + j > rowpos) s[j] = -INFINITY;
      }
      // the row maximum as a tree (exact in any order; a serial chain of dependent steps
      // would sit on the row's critical path), then the pair's
      float mt[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) mt[j] = fmaxf(s[j], s[j + 16]);
#pragma unroll
      for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) mt[j] = fmaxf(mt[j], mt[j + w]);
      float mo;
      if (!trade(i, mt[0], mo)) {
        fail = true;
        break;
      }
      const float mx = fmaxf(mt[0], mo);
      // move the reference maximum where a score passes it by more than kRescale; O and
      // l follow it. Each half rescales its O columns (warp-wide TMEM access) once every
      // P V MMA so far (tiles up to i - 1) has completed.
      const bool move = mx > m_ref + kRescale;
      const float alpha = move ? exp2f(m_ref - mx) : 1.f;   // 0 while m_ref is -inf
      if (i > 0 && __any_sync(0xffffffffu, move)) {
        if (!wait_all(&o_done[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1))) {
          fail = true;
          break;
        }
        tc::fence_after();
#pragma unroll
        for (int c = 0; c < kD / 2; c += 32) {
          float ov[32];
          tc::ld_32x32(tO + lanes + 64 * hf + c, ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] *= alpha;
          tc::st_32x32(tO + lanes + 64 * hf + c, ov);
        }
      }
      if (move) {
        l *= alpha;
        m_ref = mx;
      }
      // P buffer b is free once the P V MMAs of tile i - 2 are done
      if (i >= 2 && !wait_all(&o_done[b], (uint32_t)(((i - 2) >> 1) & 1))) {
        fail = true;
        break;
      }
      float psum[4] = {0.f, 0.f, 0.f, 0.f};   // four interleaved partial sums
      unsigned char* ph = smem + kOffPh + b * kQChunk;
      unsigned char* pl = smem + kOffPl + b * kQChunk;
#pragma unroll
      for (int c = 0; c < 4; ++c) {   // 8 keys per 16-byte piece
        float pv[8];
        // a masked score (-inf) gives 0; m_ref is finite in every row with a visible key
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float sv = s[8 * c + e];
          pv[e] = masked ? (sv == -INFINITY ? 0.f : ex2_approx(sv - m_ref)) : ex2_approx(sv - m_ref);
          psum[e & 3] += pv[e];
        }
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          hw[e] = bf2_bits(pv[2 * e], pv[2 * e + 1]);
          lw[e] = bf2_bits(pv[2 * e] - bf_lo(hw[e]), pv[2 * e + 1] - bf_hi(hw[e]));
        }
        const uint32_t o = tc::sw128_off(r, 4 * hf + c);
        *(uint4*)(ph + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *(uint4*)(pl + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      l += (psum[0] + psum[1]) + (psum[2] + psum[3]);
      fence_proxy_async_smem();
      tc::fence_before();
      mbar_arrive(&p_full[b]);
    }
    // the last tile's P V MMAs complete before O is read; the halves' sums are added in
    // the same order in both warps
    if (!fail && !wait_all(&o_done[(n_kt - 1) & 1], (uint32_t)(((n_kt - 1) >> 1) & 1))) fail = true;
    float l_other = 0.f;
    if (!fail && !trade(n_kt, l, l_other)) fail = true;
    if (fail) *(volatile int*)s_abort = 1;
    if (!fail) {   // warp-uniform; rows past the prompt load too (warp-wide) but store nothing
      tc::fence_after();
      const float lt = hf == 0 ? l + l_other : l_other + l;
      const float inv = valid ? 1.0f / lt : 0.f;
      __nv_bfloat16* out = p.out + (size_t)(valid ? row : 0) * p.Hq * kD + (size_t)h * kD + 64 * hf;
#pragma unroll
      for (int c = 0; c < kD / 2; c += 32) {
        float ov[32];
        tc::ld_32x32(tO + lanes + 64 * hf + c, ov);
        if (valid)
#pragma unroll
          for (int e = 0; e < 32; e += 8)
            *(uint4*)(out + c + e) =
                make_uint4(pack_bf(ov[e] * inv, ov[e + 1] * inv), pack_bf(ov[e + 2] * inv, ov[e + 3] * inv),
                           pack_bf(ov[e + 4] * inv, ov[e + 5] * inv), pack_bf(ov[e + 6] * inv, ov[e + 7] * inv));
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::dealloc(tbase, kTmemCols);
  }
}

// Packed copies of one kv head's keys for the kernel above: K [L][128] as is, V
// transposed to [128][L], rows past the prompt's last position zero. One CTA per 64
// keys and kv head.
__global__ void __launch_bounds__(128) prefill_kv_pack_kernel(const __nv_bfloat16* k_pages,
                                                              const __nv_bfloat16* v_pages, const int32_t* pt,
                                                              int page_size, int n_pages, int Hkv, const int32_t* pos,
                                                              int n, int cap, int L, __nv_bfloat16* ks,
                                                              __nv_bfloat16* vt, int* err) {
  __shared__ __align__(16) __nv_bfloat16 sv[kKT][kD + 8];
  const int t0 = blockIdx.x * kKT, g = blockIdx.y, tid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  // keys past the cache are never looked up (the attention kernel flags such a prompt)
  const int kv_len = min(min(pos[0] + n, cap), L);
  if (pos[0] < 0 || t0 >= kv_len) return;   // never read
  for (int i = tid; i < kKT * 16; i += 128) {
    const int r = i >> 4, c = i & 15;
    const int key = t0 + r;
    uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
    if (key < kv_len) {
      const PagedSlot sl = paged_slot(pt, key, page_size, n_pages);
      if (!sl.ok) {
        set_error(err, QD_DEVERR_PAGE);
      } else {
        const size_t off = (((size_t)sl.page * Hkv + g) * page_size + sl.slot) * kD + c * 8;
        kv = *(const uint4*)(k_pages + off);
        vv = *(const uint4*)(v_pages + off);
      }
    }
    *(uint4*)(ks + ((size_t)g * L + key) * kD + c * 8) = kv;
    *(uint4*)(&sv[r][c * 8]) = vv;
  }
  __syncthreads();
  // thread d writes V^T row d for these 64 keys (128 bytes)
  const int d = tid;
  __nv_bfloat16* dst = vt + ((size_t)g * kD + d) * L + t0;
#pragma unroll
  for (int j = 0; j < kKT; j += 8) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = (uint32_t)__bfloat16_as_ushort(sv[j + 2 * e][d]) |
             ((uint32_t)__bfloat16_as_ushort(sv[j + 2 * e + 1][d]) << 16);
    *(uint4*)(dst + j) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

size_t prefill_attention_tc_scratch_bytes(int Hkv, int cap) {
  const size_t L = ((size_t)cap + kKT - 1) / kKT * kKT;
  return 2 * (size_t)Hkv * L * kD * 2;
}

cudaError_t launch_prefill_attention_tc(const PrefillAttnArgs& a, void* scratch, size_t scratch_bytes,
                                        const Launch& L) {
  if (a.n < 1 || a.D != kD || a.Hkv < 1 || a.Hq % a.Hkv) return cudaErrorInvalidValue;
  const int cap = a.max_pages * a.page_size;
  const int Lk = (cap + kKT - 1) / kKT * kKT;
  if (!scratch || scratch_bytes < prefill_attention_tc_scratch_bytes(a.Hkv, cap)) return cudaErrorInvalidValue;
  __nv_bfloat16* ks = (__nv_bfloat16*)scratch;
  __nv_bfloat16* vt = ks + (size_t)a.Hkv * Lk * kD;
  cudaError_t e = launch_ex(prefill_kv_pack_kernel, dim3(Lk / kKT, a.Hkv), dim3(128), 0, L,
                            (const __nv_bfloat16*)a.k_pages, (const __nv_bfloat16*)a.v_pages, a.page_table,
                            a.page_size, a.n_pages, a.Hkv, a.pos, a.n, cap, Lk, ks, vt, L.err);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap tk, tv;
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  e = encode_tmap_bf16_2d(&tk, ks, (uint64_t)a.Hkv * Lk, kD, kKT);
  if (e != cudaSuccess) return e;
  e = encode_tmap_bf16_2d(&tv, vt, (uint64_t)a.Hkv * kD, (uint64_t)Lk, kD);
  if (e != cudaSuccess) return e;
  TcPfParams p = {};
  p.qkv = a.qkv; p.n = a.n; p.Hq = a.Hq; p.Hkv = a.Hkv;
  p.q_norm = (const __nv_bfloat16*)a.q_norm; p.rope = (const float2*)a.rope; p.rope_max_pos = a.rope_max_pos;
  p.eps = a.eps; p.act_bf16 = a.act_bf16; p.pos = a.pos; p.L = Lk; p.cap = cap;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.out = (__nv_bfloat16*)a.out; p.err = L.err;
  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(prefill_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(prefill_attn_tc_kernel, dim3(a.Hq, ceil_div(a.n, kQT)), dim3(kThreads), kSmem, L, tk, tv, p);
}

}  // namespace qd
