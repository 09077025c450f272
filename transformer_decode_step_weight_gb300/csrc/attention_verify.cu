// Speculative-verify attention: the k query rows of one sequence against its cached
// keys, every K/V tile read once for all of them.
//
// "qwen3-8b-rtx4080-cutedsl" README, "Speculative decoding": the target model checks
// k drafted tokens in one pass; with "Split-KV decode attention" and "GQA + QK-Norm"
// (kv head = q head / (Hq / Hkv), per-head RMSNorm of q, RoPE, partial softmax states
// combined across splits). Row i sits at position pos[i] and attends to the keys
// 0 .. pos[i]; the rows' own K/V are in the cache before this launch.
//
// GB300 layout: query column c = i * REP + h is q head g * REP + h of row i, so the
// K/V of kv head g serve k * REP columns. Grid (split, kv head); warp w owns columns
// 8w .. 8w + 7; about two CTAs per SM. K/V tiles of 64 tokens arrive by 16-byte
// cp.async in a 2-stage ring of XOR-swizzled 256-byte rows shared by the warps. Per
// warp and tile,
// S^T[64 tokens x 8 columns] = K Q^T and O^T[128 x 8] += V^T P^T run on mma.sync
// m16n8k16 (bf16 in, f32 accumulate) with q and P split into bf16 hi + lo parts, so
// scores and weights keep about 16 mantissa bits; the online softmax runs per column
// with the column's own causal limit. A split publishes (m, l, O) per column, and a
// second kernel, one CTA per (column, kv head), merges the splits in split order with
// all of a thread's loads in flight at once. Against one decode attention per row,
// the k rows no longer read the keys k times.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <algorithm>
#include <cstdlib>

namespace qd {
namespace {

constexpr int kD = 128;
constexpr int kT = 64;                   // tokens per tile
constexpr int kSt = 2;                   // ring stages
constexpr int kMaxCols = 64;             // k * REP
constexpr int kMaxWarps = kMaxCols / 8;
constexpr int kMaxSplitsV = 64;
constexpr int kTileB = kT * kD * 2;      // 16 KB per K or V tile

struct VParams {
  const float* qkv;               // f32 [k, (Hq + 2 Hkv) * 128]
  const __nv_bfloat16* q_norm;    // bf16 [128]
  const float2* rope;
  int rope_max_pos;
  float eps;
  int act_bf16;
  const int32_t* pos;             // [k]
  const int32_t* page_table;      // the sequence's page-table row
  const __nv_bfloat16* k_pages;
  const __nv_bfloat16* v_pages;
  int k, Hq, Hkv, rep, ncols, page_size, max_pages, n_pages, n_splits, chunk;
  float scale_log2;
  __nv_bfloat16* out;             // bf16 [k, Hq * 128]
  float* ws_acc;                  // [Hkv][n_splits][ncols][128]
  float* ws_ml;                   // [Hkv][n_splits][ncols][2]
  int* err;
};

QD_DEV void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
QD_DEV void ldsm_x4(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
QD_DEV void ldsm_x4_t(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// 16-byte async copy; src_bytes = 0 zero-fills the destination without reading.
QD_DEV void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
QD_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
QD_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// byte offset of (row r, 16-byte chunk c) in a swizzled 256-byte-row tile
QD_DEV uint32_t swz(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4)); }

// The K and V rows [t, t + kT) of kv head g into a stage; rows at or past t_end are
// zero-filled without reading.
QD_DEV void load_tile(const VParams& p, int g, int t, int t_end, uint32_t sK, uint32_t sV) {
  for (int i = threadIdx.x; i < kT * 16; i += blockDim.x) {
    const int r = i >> 4, c = i & 15;
    const int tok = t + r;
    const bool ok = tok < t_end;
    size_t off = 0;
    if (ok) {
      const PagedSlot sl = paged_slot(p.page_table, tok, p.page_size, p.n_pages);
      if (!sl.ok) set_error(p.err, QD_DEVERR_PAGE);
      off = (((size_t)sl.page * p.Hkv + g) * p.page_size + sl.slot) * kD + c * 8;
    }
    cp_async16(sK + swz(r, c), p.k_pages + off, ok ? 16 : 0);
    cp_async16(sV + swz(r, c), p.v_pages + off, ok ? 16 : 0);
  }
}

__global__ void __launch_bounds__(32 * kMaxWarps) verify_attn_kernel(const VParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int nw = blockDim.x >> 5;                                        // warps: 8 columns each
  unsigned char* ring = smem;                                            // kSt x (K tile, V tile)
  __nv_bfloat16* sQh = (__nv_bfloat16*)(smem + kSt * 2 * kTileB);        // [8 nw][128]
  __nv_bfloat16* sQl = sQh + nw * 8 * kD;
  __nv_bfloat16* sP = sQl + nw * 8 * kD;                                 // [warp][hi/lo][8][64]
  __shared__ int s_pos[kMaxCols];

  const int s = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();
  pdl_wait();   // the rows' K/V were written by the kernel before this one

  // every row's position must lie inside the cache and the RoPE table
  int bad = 0;
  if (tid < p.k) {
    const int ps_ = p.pos[tid];
    s_pos[tid] = ps_;
    bad = ps_ < 0 || ps_ >= p.max_pages * p.page_size || ps_ >= p.rope_max_pos;
  }
  if (__syncthreads_or(bad)) {
    if (s == 0 && tid == 0) set_error(p.err, QD_DEVERR_POS);
    return;
  }
  int lmax = 0;
  for (int i = 0; i < p.k; ++i) lmax = max(lmax, s_pos[i] + 1);
  const int n_act = (lmax + p.chunk - 1) / p.chunk;
  if (s >= n_act) return;
  const int t0 = s * p.chunk;
  const int t_end = min(t0 + p.chunk, lmax);
  const int n_tiles = (t_end - t0 + kT - 1) / kT;
  const uint32_t ring_u = smem_u32(ring);
  auto tileK = [&](int st) { return ring_u + (uint32_t)(st * 2 * kTileB); };
  auto tileV = [&](int st) { return ring_u + (uint32_t)(st * 2 * kTileB + kTileB); };
#pragma unroll
  for (int st = 0; st < kSt - 1; ++st) {
    if (st < n_tiles) load_tile(p, g, t0 + st * kT, t_end, tileK(st), tileV(st));
    cp_async_commit();
  }

  // ---- q of this warp's 8 columns: RMSNorm(q_norm), RoPE at the row's position, the
  // softmax scale (log2 e folded in), then bf16 hi + lo. Lane l holds dims l + 32e; the
  // RoPE pairs (d, d + 64) are e = 0, 2 and e = 1, 3 of the same lane.
  const int qkv_w = (p.Hq + 2 * p.Hkv) * kD;
  // the warp's 8 columns, their RoPE rows and the norm weights: every load in flight at once
  float xin[8][4];
  float2 rc[8][2];
  float qw[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) qw[e] = __bfloat162float(p.q_norm[lane + 32 * e]);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c = warp * 8 + j;
    const int row = c / p.rep, h = c - row * p.rep;
    const bool in = c < p.ncols;
    const float* src = p.qkv + (size_t)row * qkv_w + (size_t)(g * p.rep + h) * kD;
#pragma unroll
    for (int e = 0; e < 4; ++e) xin[j][e] = in ? src[lane + 32 * e] : 0.f;
    const float2* cs = p.rope + (size_t)(in ? s_pos[row] : 0) * (kD / 2);
    rc[j][0] = cs[lane];
    rc[j][1] = cs[lane + 32];
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c = warp * 8 + j;
    float qv[4] = {0.f, 0.f, 0.f, 0.f};
    if (c < p.ncols) {
      float x[4], y[4];
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[e] = xin[j][e];
        ss = fmaf(x[e], x[e], ss);
      }
      ss = warp_sum(ss);
      const float inv = 1.0f / sqrtf(ss / (float)kD + p.eps);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float n = x[e] * inv;
        if (p.act_bf16) n = round_bf16(n);
        y[e] = qw[e] * n;
        if (p.act_bf16) y[e] = round_bf16(y[e]);
      }
      const float2 c0 = rc[j][0], c1 = rc[j][1];
      qv[0] = (y[0] * c0.x - y[2] * c0.y) * p.scale_log2;   // d = lane
      qv[1] = (y[1] * c1.x - y[3] * c1.y) * p.scale_log2;   // d = lane + 32
      qv[2] = (y[2] * c0.x + y[0] * c0.y) * p.scale_log2;   // d = lane + 64
      qv[3] = (y[3] * c1.x + y[1] * c1.y) * p.scale_log2;   // d = lane + 96
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(qv[e]);
      sQh[c * kD + lane + 32 * e] = hi;
      sQl[c * kD + lane + 32 * e] = __float2bfloat16_rn(qv[e] - __bfloat162float(hi));
    }
  }
  __syncwarp();
  // B fragments of Q^T for the 8 k-steps: column n = lane / 4 of the warp's 8, dims
  // 16 ks + 2 (lane % 4) (+ 8)
  const int qn = lane >> 2, qk = (lane & 3) * 2;
  uint32_t qh[8][2], ql[8][2];
  {
    const __nv_bfloat16* qhp = sQh + (warp * 8 + qn) * kD + qk;
    const __nv_bfloat16* qlp = sQl + (warp * 8 + qn) * kD + qk;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qh[ks][0] = *(const uint32_t*)(qhp + ks * 16);
      qh[ks][1] = *(const uint32_t*)(qhp + ks * 16 + 8);
      ql[ks][0] = *(const uint32_t*)(qlp + ks * 16);
      ql[ks][1] = *(const uint32_t*)(qlp + ks * 16 + 8);
    }
  }
  // this lane's two columns of S / O: cA = 8 warp + 2 (lane % 4), cB = cA + 1, with their
  // causal limits (a padding column has none: everything masked)
  const int cA = warp * 8 + qk, cB = cA + 1;
  const int lenA = cA < p.ncols ? s_pos[cA / p.rep] + 1 : 0;
  const int lenB = cB < p.ncols ? s_pos[cB / p.rep] + 1 : 0;

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
  const int rA = (lane & 7) + ((lane >> 3) & 1) * 8, cAk = lane >> 4;        // QK ldmatrix rows / chunk
  const int rV = (lane & 7) + ((lane >> 4) & 1) * 8, cVk = (lane >> 3) & 1;  // PV ldmatrix.trans
  __nv_bfloat16* sPh = sP + warp * 2 * 8 * kT;
  __nv_bfloat16* sPl = sPh + 8 * kT;

  for (int it = 0; it < n_tiles; ++it) {
    const int st = it % kSt;
    {  // keep kSt - 1 tiles in flight (the stage refilled here was released by the
       // barrier that ended the previous iteration)
      const int nt = it + kSt - 1;
      if (nt < n_tiles) load_tile(p, g, t0 + nt * kT, t_end, tileK(nt % kSt), tileV(nt % kSt));
      cp_async_commit();
    }
    cp_async_wait<kSt - 1>();
    __syncthreads();  // every thread's copies of this tile have landed
    const int ts = t0 + it * kT;
    const uint32_t sK = tileK(st), sV = tileV(st);

    // ---- S^T = K Q^T: 4 blocks of 16 tokens x the warp's 8 columns
    float sc[4][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, sK + swz(mt * 16 + rA, 2 * ks + cAk));
        mma16816(a0, a, qh[ks][0], qh[ks][1]);
        mma16816(a1, a, ql[ks][0], ql[ks][1]);
      }
      // rows: tokens ts + 16 mt + lane / 4 (+ 8); columns cA, cB
      const int tr0 = ts + mt * 16 + (lane >> 2), tr1 = tr0 + 8;
      sc[mt][0] = tr0 < lenA ? a0[0] + a1[0] : -INFINITY;
      sc[mt][1] = tr0 < lenB ? a0[1] + a1[1] : -INFINITY;
      sc[mt][2] = tr1 < lenA ? a0[2] + a1[2] : -INFINITY;
      sc[mt][3] = tr1 < lenB ? a0[3] + a1[3] : -INFINITY;
    }

    // ---- online softmax per column (the lanes with equal lane % 4 share columns)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      mx0 = fmaxf(mx0, fmaxf(sc[mt][0], sc[mt][2]));
      mx1 = fmaxf(mx1, fmaxf(sc[mt][1], sc[mt][3]));
    }
#pragma unroll
    for (int o2 = 4; o2 <= 16; o2 <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
    const float al1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const float pv[4] = {sc[mt][0] == -INFINITY ? 0.f : exp2f(sc[mt][0] - mn0),
                           sc[mt][1] == -INFINITY ? 0.f : exp2f(sc[mt][1] - mn1),
                           sc[mt][2] == -INFINITY ? 0.f : exp2f(sc[mt][2] - mn0),
                           sc[mt][3] == -INFINITY ? 0.f : exp2f(sc[mt][3] - mn1)};
      ps0 += pv[0] + pv[2];
      ps1 += pv[1] + pv[3];
      // P^T in warp-private shared memory: [column][token] as bf16 hi + lo
      const int r0 = mt * 16 + (lane >> 2);
      const int cols[4] = {qk, qk + 1, qk, qk + 1};
      const int toks[4] = {r0, r0, r0 + 8, r0 + 8};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(pv[e]);
        sPh[cols[e] * kT + toks[e]] = hi;
        sPl[cols[e] * kT + toks[e]] = __float2bfloat16_rn(pv[e] - __bfloat162float(hi));
      }
    }
#pragma unroll
    for (int o2 = 4; o2 <= 16; o2 <<= 1) {
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, o2);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, o2);
    }
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[mt][0] *= al0;
      o[mt][1] *= al1;
      o[mt][2] *= al0;
      o[mt][3] *= al1;
    }
    __syncwarp();

    // ---- O^T += V^T P^T: 8 blocks of 16 dims x 4 blocks of 16 tokens
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      const int pi = qn * kT + kt * 16 + qk;
      const uint32_t pb0h = *(const uint32_t*)(sPh + pi), pb1h = *(const uint32_t*)(sPh + pi + 8);
      const uint32_t pb0l = *(const uint32_t*)(sPl + pi), pb1l = *(const uint32_t*)(sPl + pi + 8);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t a[4];
        ldsm_x4_t(a, sV + swz(kt * 16 + rV, 2 * mt + cVk));
        mma16816(o[mt], a, pb0h, pb1h);
        mma16816(o[mt], a, pb0l, pb1l);
      }
    }
    __syncthreads();  // the stage and the P scratch are free for the next iteration
  }
  cp_async_wait<0>();

  // O^T fragment: o[mt][0] = (dim 16 mt + lane / 4, column cA), [1] = (.., cB),
  // [2] = (dim + 8, cA), [3] = (dim + 8, cB)
  const int dA = lane >> 2;
  auto out_at = [&](int c, int d) -> __nv_bfloat16* {
    const int row = c / p.rep, h = c - row * p.rep;
    return p.out + ((size_t)row * p.Hq + g * p.rep + h) * kD + d;
  };
  if (n_act == 1) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d = mt * 16 + dA;
      if (cA < p.ncols) {
        *out_at(cA, d) = __float2bfloat16_rn(o[mt][0] / l0);
        *out_at(cA, d + 8) = __float2bfloat16_rn(o[mt][2] / l0);
      }
      if (cB < p.ncols) {
        *out_at(cB, d) = __float2bfloat16_rn(o[mt][1] / l1);
        *out_at(cB, d + 8) = __float2bfloat16_rn(o[mt][3] / l1);
      }
    }
    return;
  }

  // ---- publish this split's partial (the combine kernel merges the splits)
  const size_t base = ((size_t)g * p.n_splits + s) * p.ncols;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int d = mt * 16 + dA;
    if (cA < p.ncols) {
      p.ws_acc[(base + cA) * kD + d] = o[mt][0];
      p.ws_acc[(base + cA) * kD + d + 8] = o[mt][2];
    }
    if (cB < p.ncols) {
      p.ws_acc[(base + cB) * kD + d] = o[mt][1];
      p.ws_acc[(base + cB) * kD + d + 8] = o[mt][3];
    }
  }
  if (lane < 4) {
    if (cA < p.ncols) {
      p.ws_ml[(base + cA) * 2] = m0;
      p.ws_ml[(base + cA) * 2 + 1] = l0;
    }
    if (cB < p.ncols) {
      p.ws_ml[(base + cB) * 2] = m1;
      p.ws_ml[(base + cB) * 2 + 1] = l1;
    }
  }
}

// Merge of the splits' partials: one CTA per (column, kv head), one thread per dim;
// every split's value is loaded at once and summed in split order with the weights
// exp2(m_s - M). Nothing to do when one split covered the rows (the attention kernel
// wrote the output itself).
__global__ void __launch_bounds__(kD) verify_combine_kernel(const VParams p) {
  __shared__ float sW[kMaxSplitsV];
  __shared__ float s_tot;
  __shared__ int s_nact;
  const int c = blockIdx.x, g = blockIdx.y, d = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  const size_t slot0 = (size_t)g * p.n_splits;
  if (d < 32) {
    // the active splits (from the rows' positions, one lane each), then the weights
    // exp2(m_s - M) and the total sum of l_s weights: lane d takes splits d and d + 32,
    // summed over the lanes by a fixed butterfly
    const int cap = p.max_pages * p.page_size;
    const int ps_ = d < p.k ? p.pos[d] : 0;
    const bool bad = d < p.k && (ps_ < 0 || ps_ >= cap || ps_ >= p.rope_max_pos);
    int lm = d < p.k ? ps_ + 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lm = max(lm, __shfl_xor_sync(0xffffffffu, lm, o));
    // a row out of range: the attention kernel flagged it and wrote no partials
    const int n_act = __any_sync(0xffffffffu, bad) ? 0 : (lm + p.chunk - 1) / p.chunk;
    float mk[kMaxSplitsV / 32], lk[kMaxSplitsV / 32], M = -INFINITY;
#pragma unroll
    for (int u = 0; u < kMaxSplitsV / 32; ++u) {
      const int k = d + 32 * u;
      const bool in = k < n_act;
      mk[u] = in ? __ldcg(p.ws_ml + ((slot0 + k) * p.ncols + c) * 2) : -INFINITY;
      lk[u] = in ? __ldcg(p.ws_ml + ((slot0 + k) * p.ncols + c) * 2 + 1) : 0.f;
      M = fmaxf(M, mk[u]);
    }
    M = warp_max(M);
    float L = 0.f;
#pragma unroll
    for (int u = 0; u < kMaxSplitsV / 32; ++u) {
      const int k = d + 32 * u;
      const float wk = mk[u] == -INFINITY ? 0.f : exp2f(mk[u] - M);
      if (k < n_act) sW[k] = wk;
      L = fmaf(wk, lk[u], L);
    }
    L = warp_sum(L);
    if (d == 0) {
      s_tot = L;
      s_nact = n_act;
    }
  }
  __syncthreads();
  const int n_act = s_nact;
  if (n_act <= 1) return;   // one split wrote the output itself (or nothing to merge)
  const float* src = p.ws_acc + (slot0 * p.ncols + c) * kD + d;
  const size_t stride = (size_t)p.ncols * kD;
  constexpr int kU = 16;
  float acc = 0.f;
  for (int k0 = 0; k0 < n_act; k0 += kU) {
    float v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) v[u] = k0 + u < n_act ? __ldcg(src + (size_t)(k0 + u) * stride) : 0.f;
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (k0 + u < n_act) acc = fmaf(sW[k0 + u], v[u], acc);
  }
  const int row = c / p.rep, h = c - row * p.rep;
  p.out[((size_t)row * p.Hq + g * p.rep + h) * kD + d] = __float2bfloat16_rn(acc / s_tot);
}

constexpr size_t verify_smem_bytes(int warps) {
  return (size_t)kSt * 2 * kTileB + 2 * (size_t)warps * 8 * kD * 2 + (size_t)warps * 2 * 8 * kT * 2;
}

}  // namespace

bool verify_attention_supported(int k, int Hq, int Hkv) {
  return k >= 1 && Hkv >= 1 && Hq % Hkv == 0 && k * (Hq / Hkv) <= kMaxCols;
}

// Workspace: the decode attention's layout for B = k rows (attn_workspace_bytes(k, ..)):
// partials, then (m, l) pairs.
cudaError_t launch_verify_attention(const AttnArgs& a, int k, const Launch& L) {
  if (!verify_attention_supported(k, a.Hq, a.Hkv) || !a.qkv || !a.out_bf16) return cudaErrorInvalidValue;
  VParams p = {};
  p.qkv = a.qkv;
  p.q_norm = (const __nv_bfloat16*)a.q_norm;
  p.rope = (const float2*)a.rope;
  p.rope_max_pos = a.rope_max_pos;
  p.eps = a.eps;
  p.act_bf16 = a.act_bf16;
  p.pos = a.pos;
  p.page_table = a.page_table;   // row 0: every row of a verify pass shares the sequence's pages
  p.k_pages = (const __nv_bfloat16*)a.k_pages;
  p.v_pages = (const __nv_bfloat16*)a.v_pages;
  p.k = k; p.Hq = a.Hq; p.Hkv = a.Hkv; p.rep = a.Hq / a.Hkv; p.ncols = k * p.rep;
  p.page_size = a.page_size; p.max_pages = a.max_pages; p.n_pages = a.n_pages;
  // about two CTAs per SM over (split, kv head) (QD_VERIFY_ATTN_PER_SM), 64-token
  // multiples, at most kMaxSplitsV
  static const int per_sm = [] {
    const char* v = getenv("QD_VERIFY_ATTN_PER_SM");
    return v ? std::max(1, std::min(8, atoi(v))) : 2;
  }();
  const int ctas = per_sm * dev_info().sm_count;
  int chunk = (int)(((long long)a.max_ctx * a.Hkv + ctas - 1) / ctas);
  chunk = std::max(kT, ((chunk + kT - 1) / kT) * kT);
  while ((a.max_ctx + chunk - 1) / chunk > kMaxSplitsV) chunk += kT;
  p.chunk = chunk;
  p.n_splits = (a.max_ctx + chunk - 1) / chunk;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.out = (__nv_bfloat16*)a.out_bf16;
  // the decode attention's workspace layout for B = k (slots_cap(k, Hkv, max_ctx) slots)
  const size_t slots = (size_t)k * a.Hkv * std::min<size_t>(256, (size_t)(a.max_ctx + kT - 1) / kT);
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  unsigned char* ws = (unsigned char*)a.workspace;
  p.ws_acc = (float*)ws;
  p.ws_ml = (float*)(ws + al(slots * p.rep * kD * 4));
  p.err = L.err;
  const int warps = (p.ncols + 7) / 8;
  const size_t smem = verify_smem_bytes(warps);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(verify_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)verify_smem_bytes(kMaxWarps));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaError_t e = launch_ex(verify_attn_kernel, dim3(p.n_splits, p.Hkv), dim3(32 * warps), smem, L, p);
  if (e != cudaSuccess || p.n_splits == 1) return e;
  return launch_ex(verify_combine_kernel, dim3(p.ncols, p.Hkv), dim3(kD), 0, L, p);
}

}  // namespace qd
