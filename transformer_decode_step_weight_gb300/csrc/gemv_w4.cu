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
// GB300 layout of the work: one CTA per SM over a contiguous block of rows; a
// producer warp streams tiles of 16 rows x up to 4096 columns through a shared-
// memory ring with one TMA bulk copy per row (evict-first), issued before the
// programmatic-dependent wait, into rows padded to an odd multiple of 64 bytes so
// that the consumers' 16-byte loads hit every bank once. The multiply-add runs on
// the tensor cores (mma.sync m16n8k16, bf16 in, f32 accumulate): a 32-bit word of
// 8 nibbles gives four bf16 pairs (nibbles i and i + 4) with one shift and one bit
// operation each, (w >> 4j) & 0x000F000F | 0x43004300 = 128 + u, and one bf16x2
// subtraction of 136 makes them the codes q exactly. The activation, staged once
// in shared memory in the same pair order, is the B operand (the same in all eight
// columns), so every product q x is exact and the sums are binary32. The eight
// consumer warps split each tile's columns in 128-column chunks; partial row sums
// reduce in a fixed order through shared memory and the epilogue scales by d[r].
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

#ifndef QD_W4_WARPS
#define QD_W4_WARPS 8
#endif
#ifndef QD_W4_ONECOPY
#define QD_W4_ONECOPY 0
#endif
#ifndef QD_W4_PARTK
#define QD_W4_PARTK 4096
#endif
#ifndef QD_W4_RING_KB
#define QD_W4_RING_KB 136
#endif
constexpr int kConsW = 32 * QD_W4_WARPS;   // consumer threads
constexpr int kConsWarps = kConsW / 32;
constexpr int kTileR = 16;             // rows of a tile (the MMA's M)
constexpr int kPartK = QD_W4_PARTK;    // columns of a tile streamed per stage
constexpr int kRingW = QD_W4_RING_KB * 1024;   // ring bytes (target)
constexpr int kPhaseW = 128;           // rows reduced per window
constexpr int kMaxTopK = 16;
constexpr int kMaxTopRows = 2048;      // rows of one CTA kept for its top-k
constexpr int kMaxK = 16384;
constexpr int kMaxG = kMaxK / 8 / kConsW;   // 8-column groups of the activation per thread

struct W4Params {
  const uint8_t* W;
  const __half* d;
  int R, K, Kpad;                      // Kpad: K rounded up to 128
  int ksplit;                          // stages per tile (ceil(K / 4096))
  int rstride;                         // bytes between the rows of a stage
  int onecopy;                         // a tile's rows copied as one run (rstride = K / 2)
  int rows_base, rows_extra;
  int dsm_rows;                        // room for the scales of the CTA's rows
  int ns, stage_bytes, ring_bytes;
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

QD_DEV void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                           uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// the codes q = u - 8 of nibbles (j, j + 4) of a 32-bit word as a bf16 pair (low half:
// nibble j); 128 + u and its difference with 136 are exact in bf16
QD_DEV uint32_t nib_pair(uint32_t w, int j) {
  const uint32_t v = ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x43084308u));   // 0x4308: bf16 136
  return r;
}

QD_DEV uint32_t bf16_bits(float f) {  // f already a bf16 value
  return __float_as_uint(f) >> 16;
}

QD_DEV float silu(float g) { return g / (1.0f + expf(-g)); }

struct Cand {
  float v;
  int i;
};
QD_DEV bool better(const Cand& a, const Cand& b) { return a.v > b.v || (a.v == b.v && a.i < b.i); }

// best candidate of the consumer threads (warp shuffles, then the warps in order);
// sh: [kConsWarps] scratch; the result is valid in every consumer thread
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
  for (int w = 1; w < kConsWarps; ++w)
    if (better(sh[w], b)) b = sh[w];
  cons_sync_w();
  return b;
}

__global__ void __launch_bounds__(kConsW + 32, 1) gemv_w4_kernel(const W4Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = (uint64_t*)(smem + p.ring_bytes);
  uint64_t* empty = full + 16;
  float* red = (float*)(empty + 16);                     // [kPhaseW][kConsWarps]
  uint4* xs = (uint4*)(red + kPhaseW * kConsWarps);      // activation, bf16 pairs [Kpad / 8]
  float* dsm = (float*)(xs + p.Kpad / 8);                // the CTA's row scales [rows]
  float* keep = dsm + p.dsm_rows;                        // EPI_SWIGLU: [2 npair]; EPI_TOPK: [rows]
  __shared__ float s_ss[kConsWarps];
  __shared__ Cand s_c[kConsWarps];
  __shared__ int s_ticket;

  const int tid = threadIdx.x, lane = tid & 31;
  const int K = p.K, ns = p.ns, ksplit = p.ksplit;
  const bool pair = p.epi == EPI_SWIGLU;
  const int nown = p.rows_base + ((int)blockIdx.x < p.rows_extra ? 1 : 0);
  const int npair = pair ? nown : 0;
  const int nrows = pair ? 2 * nown : nown;
  const int r0 = (int)blockIdx.x * p.rows_base + min((int)blockIdx.x, p.rows_extra);
  const int n_tiles = (nrows + kTileR - 1) / kTileR;
  const int n_stages = n_tiles * ksplit;
  const size_t row_bytes = (size_t)K / 2;

  if (tid == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (!p.trig_late) pdl_launch_dependents();

  if (tid >= kConsW) {  // ---- producer warp: weights only, so no dependency wait
    const uint64_t pol = policy_evict_first();
    for (int i = 0; i < n_stages; ++i) {
      const int slot = i % ns;
      int ok = 1;
      if (lane == 0 && i >= ns) ok = mbar_wait_bounded(&empty[slot], (uint32_t)(((i / ns) - 1) & 1), p.err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const int tile = i / ksplit, kp = i - tile * ksplit;
      const int rows_i = min(kTileR, nrows - tile * kTileR);
      const uint32_t bytes = (uint32_t)(min(K - kp * kPartK, kPartK) / 2);
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)rows_i * bytes);
      __syncwarp();
      unsigned char* dst0 = ring + (size_t)slot * p.stage_bytes;
      if (p.onecopy) {  // contiguous rows: one copy per run (two where gate rows end)
        if (lane == 0) {
          const int a = tile * kTileR;
          const int na = pair ? max(0, min(a + rows_i, npair) - a) : rows_i;
          auto copy = [&](void* dd, const void* src, uint32_t n) {
            if (p.w_evict_first) bulk_g2s_hint(dd, src, n, &full[slot], pol);
            else bulk_g2s(dd, src, n, &full[slot]);
          };
          if (na > 0) copy(dst0, p.W + ((size_t)r0 + a) * row_bytes, (uint32_t)(na * row_bytes));
          if (rows_i > na)
            copy(dst0 + (size_t)na * row_bytes, p.W + ((size_t)p.pair_F + r0 + a + na - npair) * row_bytes,
                 (uint32_t)((rows_i - na) * row_bytes));
        }
      } else if (lane < rows_i) {  // one row per lane; the SwiGLU form's up rows follow the gate rows
        const int lr = tile * kTileR + lane;
        const size_t row = (pair && lr >= npair) ? (size_t)p.pair_F + r0 + (lr - npair) : (size_t)r0 + lr;
        const unsigned char* src = p.W + row * row_bytes + (size_t)kp * (kPartK / 2);
        unsigned char* dst = dst0 + (size_t)lane * p.rstride;
        if (p.w_evict_first) bulk_g2s_hint(dst, src, bytes, &full[slot], pol);
        else bulk_g2s(dst, src, bytes, &full[slot]);
      }
    }
    __syncwarp();
    pdl_launch_dependents();
    l2_prefetch_spans(p.pf, blockIdx.x, gridDim.x, lane);
    return;
  }

  // ---- consumers: the activation, once, as bf16 pairs in shared memory. Group G of
  // 8 columns (k = 8G .. 8G + 7) is stored at ((c * 4 + w) * 4 + t), c = G / 16,
  // t = (G / 4) % 4, w = G % 4, as the pairs (k, k + 4) for k = 8G .. 8G + 3: the
  // B-operand registers of lane t for word w of its 32 columns of chunk c.
  const int NG = p.Kpad / 8, NGK = K / 8;
  for (int lr = tid; lr < nrows; lr += kConsW) {   // row scales (weights: before the dependency wait)
    const size_t row = (pair && lr >= npair) ? (size_t)p.pair_F + r0 + (lr - npair) : (size_t)r0 + lr;
    dsm[lr] = __half2float(p.d[row]);
  }
  uint4 wn[kMaxG];
#pragma unroll
  for (int j = 0; j < kMaxG; ++j) {
    const int G = tid + j * kConsW;
    wn[j] = (p.pro == PRO_RMSNORM && G < NGK) ? *(const uint4*)(p.norm_w + 8 * G) : make_uint4(0u, 0u, 0u, 0u);
  }
  pdl_wait();
  float xv[kMaxG][8];
#pragma unroll
  for (int j = 0; j < kMaxG; ++j) {
    const int G = tid + j * kConsW;
#pragma unroll
    for (int e = 0; e < 8; ++e) xv[j][e] = 0.f;
    if (G >= NGK) continue;
    if (p.pro == PRO_X_BF16) {
      const uint4 v = *(const uint4*)((const __nv_bfloat16*)p.x + 8 * G);
      xv[j][0] = bf_lo(v.x); xv[j][1] = bf_hi(v.x); xv[j][2] = bf_lo(v.y); xv[j][3] = bf_hi(v.y);
      xv[j][4] = bf_lo(v.z); xv[j][5] = bf_hi(v.z); xv[j][6] = bf_lo(v.w); xv[j][7] = bf_hi(v.w);
    } else {  // PRO_X_F32 or PRO_RMSNORM: f32 source
      const float4 a = *(const float4*)((const float*)p.x + 8 * G);
      const float4 b = *(const float4*)((const float*)p.x + 8 * G + 4);
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
    if (lane == 0) s_ss[tid >> 5] = ss;
    cons_sync_w();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kConsWarps; ++i) tot += s_ss[i];
    const float inv = 1.0f / sqrtf(tot / (float)K + p.eps);
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
    const int G = tid + j * kConsW;
    if (G >= NG) continue;
    uint4 v;
    v.x = bf16_bits(xv[j][0]) | (bf16_bits(xv[j][4]) << 16);
    v.y = bf16_bits(xv[j][1]) | (bf16_bits(xv[j][5]) << 16);
    v.z = bf16_bits(xv[j][2]) | (bf16_bits(xv[j][6]) << 16);
    v.w = bf16_bits(xv[j][3]) | (bf16_bits(xv[j][7]) << 16);
    xs[((G >> 4) * 4 + (G & 3)) * 4 + ((G >> 2) & 3)] = v;
  }
  cons_sync_w();

  const bool topk = p.epi == EPI_TOPK;
  auto epilogue = [&](int lr, float s) {  // lr: local row of the CTA, s: sum q x of it
    if (pair) {
      keep[lr] = s;
      return;
    }
    const int r = r0 + lr;
    const float v = dsm[lr] * s;
    if (p.epi == EPI_RESID_ADD) {
      p.y[r] += v;
    } else {
      p.y[r] = v;
      if (topk) keep[lr] = v;
    }
  };

  // ---- main loop: lane (g, t) of warp wp holds rows g and g + 8 of the tile; per
  // 128-column chunk it takes 32 columns (t * 32 ..) of each: 4 words, 8 MMAs
  const int wp = tid >> 5, g = lane >> 2, t = lane & 3;
  float acc[4][4];
#pragma unroll
  for (int w = 0; w < 4; ++w)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[w][e] = 0.f;
  int ph_base = 0;
  for (int i = 0; i < n_stages; ++i) {
    const int slot = i % ns;
    if (!mbar_wait_bounded(&full[slot], (uint32_t)((i / ns) & 1), p.err)) {
      for (int k = 1; k < ns && i + k < n_stages; ++k)
        mbar_wait_bounded(&full[(i + k) % ns], (uint32_t)(((i + k) / ns) & 1), p.err);
      return;
    }
    if (i + 1 == n_stages) pdl_launch_dependents();
    const int tile = i / ksplit, kp = i - tile * ksplit;
    const int nch = (min(K - kp * kPartK, kPartK) + 127) >> 7;
    const unsigned char* base = ring + (size_t)slot * p.stage_bytes + (size_t)g * p.rstride + 16 * t;
    for (int ch = wp; ch < nch; ch += kConsWarps) {
      const uint4* xq = xs + (size_t)(kp * (kPartK / 128) + ch) * 16 + t;
      const uint4 wa = *(const uint4*)(base + 64 * ch);
      const uint4 wb = *(const uint4*)(base + 8 * (size_t)p.rstride + 64 * ch);
      const uint32_t ra[4] = {wa.x, wa.y, wa.z, wa.w}, rb[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint4 xb = xq[4 * w];
        mma_bf16_16816(acc[w], nib_pair(ra[w], 0), nib_pair(rb[w], 0), nib_pair(ra[w], 1), nib_pair(rb[w], 1),
                       xb.x, xb.y);
        mma_bf16_16816(acc[w], nib_pair(ra[w], 2), nib_pair(rb[w], 2), nib_pair(ra[w], 3), nib_pair(rb[w], 3),
                       xb.z, xb.w);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (kp + 1 < ksplit) continue;
    // the tile's partial sums of this warp: row g in acc[.][0], row g + 8 in acc[.][2]
    const float sg = (acc[0][0] + acc[1][0]) + (acc[2][0] + acc[3][0]);
    const float sg8 = (acc[0][2] + acc[1][2]) + (acc[2][2] + acc[3][2]);
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[w][e] = 0.f;
    const int lr = tile * kTileR + g;
    if (t == 0) {
      if (lr < nrows) red[(lr - ph_base) * kConsWarps + wp] = sg;
      if (lr + 8 < nrows) red[(lr + 8 - ph_base) * kConsWarps + wp] = sg8;
    }
    const int done = min((tile + 1) * kTileR, nrows);
    if (done + kTileR - ph_base > kPhaseW || i + 1 == n_stages) {
      const int nph = done - ph_base;
      cons_sync_w();
      for (int r = tid; r < nph; r += kConsW) {
        float a = 0.f;
#pragma unroll
        for (int k = 0; k < kConsWarps; ++k) a += red[r * kConsWarps + k];
        epilogue(ph_base + r, a);
      }
      cons_sync_w();
      ph_base = done;
    }
  }
  if (pair) {  // h = bf16(silu(gate) * up) of the CTA's pairs
    for (int j = tid; j < npair; j += kConsW) {
      const float gv = dsm[j] * keep[j];
      const float uv = dsm[npair + j] * keep[npair + j];
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

cudaError_t launch_w4(const W4Params& p, int grid, size_t smem, const Launch& L) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemv_w4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         dev_info().max_smem_optin - 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(gemv_w4_kernel, dim3(grid), dim3(kConsW + 32), smem, L, p);
}

}  // namespace

bool gemv_w4_supported(int K) { return K >= 32 && K % 32 == 0 && K <= kMaxK; }

// candidates [SMs][kMaxTopK] (value, row) and the merge ticket
size_t w4_topk_workspace_bytes() {
  return (((size_t)dev_info().sm_count * kMaxTopK * 8 + 255) & ~(size_t)255) + 256;
}

cudaError_t launch_gemv_w4(const GemvW4Args& a, const Launch& L) {
  // K a multiple of 256: the tcgen05 form (gemv_w4_tc.cu); this form covers the rest
  if (gemv_w4_tc_supported(a.K)) return launch_gemv_w4_tc(a, a.split_ws, a.split_ws_bytes, L);
  if (!gemv_w4_supported(a.K) || a.R < 1) return cudaErrorInvalidValue;
  const bool pair = a.epi == EPI_SWIGLU, topk = a.epi == EPI_TOPK;
  if (pair && a.R % 2) return cudaErrorInvalidValue;
  if (topk && (a.top_k < 1 || a.top_k > kMaxTopK || !a.ws)) return cudaErrorInvalidValue;
  W4Params p = {};
  p.W = (const uint8_t*)a.W;
  p.d = (const __half*)a.d;
  p.R = a.R; p.K = a.K;
  p.Kpad = ceil_div(a.K, 128) * 128;
  p.ksplit = ceil_div(a.K, kPartK);
  const int part_max = std::min(p.Kpad, kPartK);
  p.rstride = ceil_div(part_max / 2, 128) * 128 + 64;   // an odd multiple of 64 bytes
  p.onecopy = QD_W4_ONECOPY && p.ksplit == 1 && a.K % 128 == 0;
  if (p.onecopy) p.rstride = a.K / 2;
  p.stage_bytes = ceil_div(kTileR * p.rstride, 128) * 128;
  p.ns = std::max(2, std::min(8, kRingW / p.stage_bytes));
  p.ring_bytes = p.ns * p.stage_bytes;
  const int units = pair ? a.R / 2 : a.R;
  const int grid = std::max(1, std::min(units, dev_info().sm_count));
  p.rows_base = units / grid; p.rows_extra = units % grid;
  p.dsm_rows = (pair ? 2 : 1) * (p.rows_base + 1);
  if (topk && p.rows_base + 1 > kMaxTopRows) return cudaErrorInvalidValue;
  p.pair_F = pair ? a.R / 2 : 0;
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
  size_t smem = (size_t)p.ring_bytes + 32 * 8 + (size_t)kPhaseW * kConsWarps * 4 + (size_t)p.Kpad * 2 +
                ((size_t)p.dsm_rows + keep_floats) * 4;
  if (smem > (size_t)dev_info().max_smem_optin - 2048) return cudaErrorInvalidValue;
  smem = std::max(smem, (size_t)dev_info().max_smem_optin / 2 + 1024);  // one GEMV CTA per SM
  return launch_w4(p, grid, smem, L);
}

}  // namespace qd
