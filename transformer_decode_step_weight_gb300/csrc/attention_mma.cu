// GQA split-KV decode attention on the tensor cores (bf16 MMA, f32 accumulate),
// with the per-head QK RMSNorm, RoPE and K/V cache write of the current token
// fused in.
//
// Same computation and split/combine protocol as the CUDA-core form in
// attention.cu ("qwen3-8b-rtx4080-cutedsl" README, "Split-KV decode attention"
// and "GQA + QK-Norm": the q heads sharing a kv head are packed into one CTA,
// turning their dot products into a small matrix product; "GPU Kernel Lab"
// README, "Decode integration"). Here both contractions of a 64-token tile are
// warp-level MMAs:
//   * S^T[16 tokens x 8 heads] = K[16 x 128] . Q^T[128 x 8] per warp, q split
//     into bf16 hi + lo parts (two MMAs), so scores keep ~16 mantissa bits;
//   * an online softmax per warp over its 16 tokens (running max and sum per
//     head, registers only);
//   * O^T[128 dims x 8 heads] += V^T[128 x 16] . P^T[16 x 8], P split into
//     bf16 hi + lo, V read with transposing ldmatrix;
//   * K/V tiles arrive by 16-byte cp.async into a 2- or 4-stage ring whose rows are
//     XOR-swizzled (16-byte chunk c of row r at c ^ (r & 7)), so every ldmatrix
//     is bank-conflict free; rows past the sequence are zero-filled.
// Heads beyond REP are zero padding (never stored). At the end the four warps'
// (max, sum, O) merge in shared memory and the split publishes its partial for
// the ticketed combine (or writes the result when it is the only split).
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <algorithm>
#include <cstdlib>
#include <cstring>

namespace qd {
namespace {

constexpr int kD = 128;
constexpr int kT = 64;                 // tokens per tile
constexpr int kW = 4;                  // warps (16 tokens each)
constexpr int kTh = kW * 32;           // == kD: one thread per head dimension in the prologue
constexpr int kHP = 8;                 // heads padded to the MMA N
constexpr int kMaxSplitsM = 256;
constexpr int kTileBytes = kT * kD * 2;  // 16 KB per K or V tile
constexpr float kLog2e = 1.4426950408889634f;

struct MParams {
  const float* q;
  const float* qkv;
  const __nv_bfloat16* q_norm;
  const __nv_bfloat16* k_norm;
  const float2* rope;
  int rope_max_pos;
  float eps;
  int act_bf16;
  const int32_t* pos;
  const int32_t* seq_lens;
  const __nv_bfloat16* k_pages;
  const __nv_bfloat16* v_pages;
  __nv_bfloat16* k_pages_w;
  __nv_bfloat16* v_pages_w;
  const int32_t* page_table;
  int B, Hq, Hkv, page_size, max_pages, n_pages, n_splits, chunk;
  float scale_log2;
  float* out_f32;
  __nv_bfloat16* out_bf16;
  float* ws_acc;
  float* ws_ml;
  int* ws_cnt;
  int* err;
  int trig_late;
  int kv_ready;
};

// ---- warp-level MMA / ldmatrix / cp.async wrappers
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
// the TMA form keeps each 128-byte half of the rows in its own 8 KB block, in
// the 128-byte swizzle the copy engine writes (chunk c of row r at c ^ (r & 7))
QD_DEV uint32_t swz_tma(int r, int c) {
  return (uint32_t)((c >> 3) * (kT * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}
template <bool TMA>
QD_DEV uint32_t swz_t(int r, int c) { return TMA ? swz_tma(r, c) : swz(r, c); }

// Issue the cp.async copies of one tile's K and V rows [t, t + kT) (rows at or
// past t_valid_end are zero-filled, rows of the current token are skipped and
// later written from registers).
QD_DEV void load_tile(const MParams& p, int b, int g, int t, int t_valid_end, int skip_tok, uint32_t sK,
                      uint32_t sV) {
  const int ps = p.page_size;
  const int32_t* pt = p.page_table + (size_t)b * p.max_pages;
#pragma unroll
  for (int j = 0; j < (kT * 16) / kTh; ++j) {
    const int i = threadIdx.x + j * kTh;
    const int r = i >> 4, c = i & 15;
    const int tok = t + r;
    const bool ok = tok < t_valid_end && tok != skip_tok;
    size_t off = 0;
    if (ok) {
      const PagedSlot sl = paged_slot(pt, tok, ps, p.n_pages);
      if (!sl.ok) set_error(p.err, QD_DEVERR_PAGE);
      off = (((size_t)sl.page * p.Hkv + g) * ps + sl.slot) * kD + c * 8;
    }
    cp_async16(sK + swz(r, c), p.k_pages + off, ok ? 16 : 0);
    cp_async16(sV + swz(r, c), p.v_pages + off, ok ? 16 : 0);
  }
}

QD_DEV void tma_box(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// One warp's share of a tile: the 16-row page segment of K and of V starting at token
// tok0 (two 64-column boxes each) onto the warp's own barrier; a segment at or past
// t_valid_end is not copied and the barrier completes on the arrival alone.
QD_DEV void load_seg_tma(const MParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV, int b, int g, int tok0,
                         int t_valid_end, uint32_t dk, uint32_t dv, uint64_t* bar) {
  if (tok0 >= t_valid_end) {
    mbar_arrive(bar);
    return;
  }
  const PagedSlot sl = paged_slot(p.page_table + (size_t)b * p.max_pages, tok0, p.page_size, p.n_pages);
  if (!sl.ok) set_error(p.err, QD_DEVERR_PAGE);
  const int row = (sl.page * p.Hkv + g) * p.page_size + sl.slot;
  mbar_arrive_expect_tx(bar, 4 * 16 * 128);
  tma_box(dk, tmK, 0, row, bar);
  tma_box(dk + kT * 128, tmK, 64, row, bar);
  tma_box(dv, tmV, 0, row, bar);
  tma_box(dv + kT * 128, tmV, 64, row, bar);
}

template <int REP, bool FUSED, int kSt, bool TMA>
__global__ void __launch_bounds__(kTh) attn_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                                                       const __grid_constant__ CUtensorMap tmV, const MParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // 1024-byte alignment for the swizzled TMA boxes
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* ring = smem;                                         // kSt x (K, V) tiles
  __nv_bfloat16* sQh = (__nv_bfloat16*)(smem + kSt * 2 * kTileBytes);  // [8][128]
  __nv_bfloat16* sQl = sQh + kHP * kD;
  __nv_bfloat16* sP = sQl + kHP * kD;                                  // [warp][hi/lo][8][16]
  float* sQf = (float*)(sP + kW * 2 * kHP * 16);                       // [REP][128] f32 staging
  float* sM = sQf + REP * kD;                                          // [kW][8]
  float* sL = sM + kW * kHP;                                           // [kW][8]
  float* sRed = sL + kW * kHP;                                         // scratch [4][REP + 1]
  // TMA: full[kSt][kW], one barrier per stage and warp (each warp loads and reads its
  // own 16-token segment of every tile, so the warps never wait for one another)
  uint64_t* bars = (uint64_t*)(((uintptr_t)(sRed + 4 * 9) + 7) & ~(uintptr_t)7);
  __shared__ int s_ticket;
  __shared__ int s_fail;
  __shared__ float s_x[kD];
  __shared__ __align__(16) __nv_bfloat16 s_knew[kD];
  __shared__ __align__(16) __nv_bfloat16 s_vnew[kD];

  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (!p.trig_late) pdl_launch_dependents();

  // The position (or length), the page table and the cached rows below it are
  // final before this kernel starts (only q, k, v come from the kernel it waits
  // on), so the first K/V tiles are requested before the dependency wait.
  const int pv_raw = FUSED ? p.pos[b] : p.seq_lens[b];
  int len, pos = 0;
  if (FUSED) {
    pos = pv_raw;
    len = pos + 1;
  } else {
    len = pv_raw;
  }
  const int cap = p.max_pages * p.page_size;
  if (len < 0 || len > cap || (FUSED && (pos < 0 || pos >= p.rope_max_pos))) {
    if (s == 0 && tid == 0) set_error(p.err, QD_DEVERR_POS);
    pdl_launch_dependents();
    return;
  }
  const size_t head0 = (size_t)b * p.Hq + g * REP;
  if (len == 0) {  // empty sequence (standalone form only): zero output
    pdl_wait();
    if (s == 0 && !FUSED)
      for (int e = tid; e < REP * kD; e += kTh) p.out_f32[head0 * kD + e] = 0.f;
    return;
  }
  const int n_act = (len + p.chunk - 1) / p.chunk;
  if (s >= n_act) return;
  const int t0 = s * p.chunk;
  const int t_end = min(t0 + p.chunk, len);
  const int n_tiles = (t_end - t0 + kT - 1) / kT;
  const int skip_tok = (FUSED && !p.kv_ready) ? pos : -1;   // the current token comes from registers
  const uint32_t ring_u = smem_u32(ring);
  auto tileK = [&](int st) { return ring_u + (uint32_t)(st * 2 * kTileBytes); };
  auto tileV = [&](int st) { return ring_u + (uint32_t)(st * 2 * kTileBytes + kTileBytes); };

  // ---- start streaming the first tiles, then wait for and build q (and the new k, v)
  if constexpr (TMA) {
    if (tid == 0) {
      for (int e = 0; e < kSt * kW; ++e) mbar_init(&bars[e], 1);
      fence_mbar_init();
      s_fail = 0;
    }
    __syncthreads();  // the barriers are initialised before anyone issues or waits
    if (lane == 0)
      for (int st = 0; st < kSt - 1 && st < n_tiles; ++st)
        load_seg_tma(p, &tmK, &tmV, b, g, t0 + st * kT + 16 * warp, t_end, tileK(st) + warp * 16 * 128,
                     tileV(st) + warp * 16 * 128, &bars[st * kW + warp]);
  } else {
#pragma unroll
    for (int st = 0; st < kSt - 1; ++st) {
      if (st < n_tiles) load_tile(p, b, g, t0 + st * kT, t_end, skip_tok, tileK(st), tileV(st));
      cp_async_commit();
    }
  }
  pdl_wait();
  const int qkv_w = (p.Hq + 2 * p.Hkv) * kD;
  float xq[REP], xk = 0.f, xvv = 0.f;
  if (FUSED) {
    const float* qkv = p.qkv + (size_t)b * qkv_w;
#pragma unroll
    for (int i = 0; i < REP; ++i) xq[i] = qkv[(g * REP + i) * kD + tid];
    xk = qkv[(p.Hq + g) * kD + tid];
    xvv = qkv[(p.Hq + p.Hkv + g) * kD + tid];
  } else {
#pragma unroll
    for (int i = 0; i < REP; ++i) xq[i] = p.q[((size_t)b * p.Hq + g * REP + i) * kD + tid];
  }

  float k_new = 0.f, v_new = 0.f;
  const bool own_pos = FUSED && !p.kv_ready && pos >= t0 && pos < t_end;
  if (FUSED) {
    const float2 cs = p.rope[(size_t)pos * (kD / 2) + (tid & 63)];
    float xv[REP + 1];
#pragma unroll
    for (int i = 0; i < REP; ++i) xv[i] = xq[i];
    xv[REP] = own_pos ? xk : 0.f;
    const float vx = own_pos ? xvv : 0.f;
#pragma unroll
    for (int i = 0; i <= REP; ++i) {
      const float ss = warp_sum(xv[i] * xv[i]);
      if (lane == 0) sRed[warp * (REP + 1) + i] = ss;
    }
    __syncthreads();
    float y[REP + 1];
#pragma unroll
    for (int i = 0; i <= REP; ++i) {
      const float tot = (sRed[i] + sRed[(REP + 1) + i]) + (sRed[2 * (REP + 1) + i] + sRed[3 * (REP + 1) + i]);
      const float inv = 1.0f / sqrtf(tot / (float)kD + p.eps);
      float n = xv[i] * inv;
      if (p.act_bf16) n = round_bf16(n);
      const __nv_bfloat16* w = i < REP ? p.q_norm : p.k_norm;
      y[i] = __bfloat162float(w[tid]) * n;
      if (p.act_bf16) y[i] = round_bf16(y[i]);
      if (i < REP) sQf[i * kD + tid] = y[i];
      else s_x[tid] = y[i];
    }
    __syncthreads();
    float r[REP + 1];
#pragma unroll
    for (int i = 0; i <= REP; ++i) {
      const float other = i < REP ? sQf[i * kD + (tid ^ 64)] : s_x[tid ^ 64];
      r[i] = (tid < 64) ? (y[i] * cs.x - other * cs.y) : (y[i] * cs.x + other * cs.y);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < REP; ++i) sQf[i * kD + tid] = r[i] * p.scale_log2;
    if (own_pos) {
      k_new = round_bf16(r[REP]);
      v_new = round_bf16(vx);
      s_knew[tid] = __float2bfloat16_rn(k_new);
      s_vnew[tid] = __float2bfloat16_rn(v_new);
      const PagedSlot own = paged_slot(p.page_table + (size_t)b * p.max_pages, pos, p.page_size, p.n_pages);
      if (!own.ok) {
        if (tid == 0) set_error(p.err, QD_DEVERR_PAGE);
      } else {
        const size_t off = (((size_t)own.page * p.Hkv + g) * p.page_size + own.slot) * kD + tid;
        p.k_pages_w[off] = __float2bfloat16_rn(k_new);
        p.v_pages_w[off] = __float2bfloat16_rn(v_new);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < REP; ++i) sQf[i * kD + tid] = xq[i] * p.scale_log2;
  }
  __syncthreads();
  // q as bf16 hi + lo, heads padded to 8 with zeros
#pragma unroll
  for (int h = 0; h < kHP; ++h) {
    const float qv = h < REP ? sQf[h * kD + tid] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(qv);
    sQh[h * kD + tid] = hi;
    sQl[h * kD + tid] = __float2bfloat16_rn(qv - __bfloat162float(hi));
  }
  __syncthreads();

  // B fragments of Q^T for the 8 k-steps: head n = lane / 4, dims 16ks + 2(lane % 4) (+8)
  const int qn = lane >> 2, qk = (lane & 3) * 2;
  uint32_t qh[8][2], ql[8][2];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    qh[ks][0] = *(const uint32_t*)(sQh + qn * kD + ks * 16 + qk);
    qh[ks][1] = *(const uint32_t*)(sQh + qn * kD + ks * 16 + qk + 8);
    ql[ks][0] = *(const uint32_t*)(sQl + qn * kD + ks * 16 + qk);
    ql[ks][1] = *(const uint32_t*)(sQl + qn * kD + ks * 16 + qk + 8);
  }

  // per-thread running state for heads h0 = 2(lane % 4), h0 + 1
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;

  const int rA = (lane & 7) + ((lane >> 3) & 1) * 8, cA = lane >> 4;        // QK ldmatrix rows / chunk
  const int rV = (lane & 7) + ((lane >> 4) & 1) * 8, cV = (lane >> 3) & 1;  // PV ldmatrix.trans
  __nv_bfloat16* sPh = sP + warp * 2 * kHP * 16;
  __nv_bfloat16* sPl = sPh + kHP * 16;

  for (int it = 0; it < n_tiles; ++it) {
    const int st = it % kSt;
    const int ts = t0 + it * kT;
    if constexpr (TMA) {
      const int nt = it + kSt - 1;   // keep kSt - 1 tiles in flight, this warp's segments only
      if (lane == 0 && nt < n_tiles) {
        fence_proxy_async_smem();    // the warp's earlier reads and writes of the stage come first
        load_seg_tma(p, &tmK, &tmV, b, g, t0 + nt * kT + 16 * warp, t_end, tileK(nt % kSt) + warp * 16 * 128,
                     tileV(nt % kSt) + warp * 16 * 128, &bars[(nt % kSt) * kW + warp]);
      }
      const bool got = mbar_wait_bounded(&bars[st * kW + warp], (uint32_t)((it / kSt) & 1), p.err);
      if (!__all_sync(0xffffffffu, got)) {  // a copy never arrived: let this warp's others land, then stop
        for (int k = 1; k < kSt && it + k < n_tiles; ++k)
          mbar_wait_bounded(&bars[((it + k) % kSt) * kW + warp], (uint32_t)(((it + k) / kSt) & 1), p.err);
        if (lane == 0) s_fail = 1;
        break;
      }
      unsigned char* sVg = ring + st * 2 * kTileBytes + kTileBytes;
      const int rw = warp * 16;      // this warp's rows of the tile
      if (ts + rw + 16 > t_end) {    // its rows past the sequence: V zeroed (K rows are masked)
        const int r_lo = max(rw, t_end - ts);
        for (int e = lane; e < (rw + 16 - r_lo) * 16; e += 32) {
          const int r = r_lo + (e >> 4), c = e & 15;
          *(uint4*)(sVg + swz_tma(r, c)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (own_pos && pos >= ts + rw && pos < ts + rw + 16) {  // the current token's row, from registers
        const int r = pos - ts;
        const int d0 = 4 * lane;
        const uint32_t o16 = swz_tma(r, d0 >> 3) + (uint32_t)((d0 & 7) * 2);
        *(uint2*)(ring + st * 2 * kTileBytes + o16) = *(const uint2*)(s_knew + d0);
        *(uint2*)(sVg + o16) = *(const uint2*)(s_vnew + d0);
      }
      __syncwarp();
    } else {
      {  // keep kSt - 1 tiles in flight
        const int nt = it + kSt - 1;
        if (nt < n_tiles) load_tile(p, b, g, t0 + nt * kT, t_end, skip_tok, tileK(nt % kSt), tileV(nt % kSt));
        cp_async_commit();
      }
      cp_async_wait<kSt - 1>();
      __syncthreads();  // every thread's copies of this tile have landed
      if (own_pos && pos >= ts && pos < ts + kT) {  // the current token's row, swizzled like the copies
        const int r = pos - ts;
        const uint32_t o16 = swz(r, tid >> 3) + (uint32_t)((tid & 7) * 2);
        *(__nv_bfloat16*)(ring + st * 2 * kTileBytes + o16) = __float2bfloat16_rn(k_new);
        *(__nv_bfloat16*)(ring + st * 2 * kTileBytes + kTileBytes + o16) = __float2bfloat16_rn(v_new);
        __syncthreads();
      }
    }

    // ---- S^T = K . Q^T for this warp's 16 tokens
    const uint32_t sK = tileK(st), sV = tileV(st);
    float sc[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};  // two independent MMA chains
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a[4];
      ldsm_x4(a, sK + swz_t<TMA>(warp * 16 + rA, 2 * ks + cA));
      mma16816(sc, a, qh[ks][0], qh[ks][1]);
      mma16816(sl, a, ql[ks][0], ql[ks][1]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[e] += sl[e];
    // rows: tokens tr0 = ts + 16w + lane/4, tr1 = tr0 + 8; cols: heads 2(lane%4), +1
    const int tr0 = ts + warp * 16 + (lane >> 2), tr1 = tr0 + 8;
    if (tr0 >= t_end) { sc[0] = -INFINITY; sc[1] = -INFINITY; }
    if (tr1 >= t_end) { sc[2] = -INFINITY; sc[3] = -INFINITY; }

    // ---- online softmax over this warp's tokens (lanes with equal lane%4 share heads)
    float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
    for (int o2 = 4; o2 <= 16; o2 <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
    const float al1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
    const float p00 = sc[0] == -INFINITY ? 0.f : exp2f(sc[0] - mn0);
    const float p01 = sc[1] == -INFINITY ? 0.f : exp2f(sc[1] - mn1);
    const float p10 = sc[2] == -INFINITY ? 0.f : exp2f(sc[2] - mn0);
    const float p11 = sc[3] == -INFINITY ? 0.f : exp2f(sc[3] - mn1);
    float ps0 = p00 + p10, ps1 = p01 + p11;
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

    // ---- P^T through warp-private shared memory: [head][token] as bf16 hi + lo
    {
      const int h0 = (lane & 3) * 2, r0 = lane >> 2;
      const float pv[4] = {p00, p01, p10, p11};
      const int hh[4] = {h0, h0 + 1, h0, h0 + 1};
      const int rr[4] = {r0, r0, r0 + 8, r0 + 8};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(pv[e]);
        sPh[hh[e] * 16 + rr[e]] = hi;
        sPl[hh[e] * 16 + rr[e]] = __float2bfloat16_rn(pv[e] - __bfloat162float(hi));
      }
    }
    __syncwarp();
    const uint32_t pb0h = *(const uint32_t*)(sPh + qn * 16 + qk), pb1h = *(const uint32_t*)(sPh + qn * 16 + qk + 8);
    const uint32_t pb0l = *(const uint32_t*)(sPl + qn * 16 + qk), pb1l = *(const uint32_t*)(sPl + qn * 16 + qk + 8);

    // ---- O^T += V^T . P^T over this warp's 16 tokens, 8 tiles of 16 dims
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t a[4];
      ldsm_x4_t(a, sV + swz_t<TMA>(warp * 16 + rV, 2 * mt + cV));
      mma16816(o[mt], a, pb0h, pb1h);
      mma16816(o[mt], a, pb0l, pb1l);
    }
    __syncwarp();
    if constexpr (!TMA) __syncthreads();  // the stage is refilled by the next iteration's copies
  }
  if constexpr (!TMA) {
    cp_async_wait<0>();
  } else {
    __syncthreads();  // every warp has left the ring, its copies all landed, before the ring is reused
    if (s_fail) return;
  }
  pdl_launch_dependents();

  // ---- merge the four warps: O^T fragments -> [warp][head][dim] f32 (ring is idle now)
  float* sO = (float*)ring;
  {
    const int h0 = (lane & 3) * 2, d0 = lane >> 2;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      sO[(warp * kHP + h0) * kD + mt * 16 + d0] = o[mt][0];
      sO[(warp * kHP + h0 + 1) * kD + mt * 16 + d0] = o[mt][1];
      sO[(warp * kHP + h0) * kD + mt * 16 + d0 + 8] = o[mt][2];
      sO[(warp * kHP + h0 + 1) * kD + mt * 16 + d0 + 8] = o[mt][3];
    }
    if (lane < 4) {
      sM[warp * kHP + h0] = m0;
      sM[warp * kHP + h0 + 1] = m1;
      sL[warp * kHP + h0] = l0;
      sL[warp * kHP + h0 + 1] = l1;
    }
  }
  __syncthreads();
  float oo[REP], MM[REP], LL[REP];
#pragma unroll
  for (int h = 0; h < REP; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kW; ++w) M = fmaxf(M, sM[w * kHP + h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const float c = sM[w * kHP + h] == -INFINITY ? 0.f : exp2f(sM[w * kHP + h] - M);
      L = fmaf(c, sL[w * kHP + h], L);
      O = fmaf(c, sO[(w * kHP + h) * kD + tid], O);
    }
    oo[h] = O;
    MM[h] = M;
    LL[h] = L;
  }

  if (n_act == 1) {
#pragma unroll
    for (int h = 0; h < REP; ++h) {
      const float r = oo[h] / LL[h];
      if (p.out_bf16) p.out_bf16[(head0 + h) * kD + tid] = __float2bfloat16_rn(r);
      else p.out_f32[(head0 + h) * kD + tid] = r;
    }
    return;
  }

  // ---- publish the partial, take a ticket; the last split combines in split order
  const size_t slot0 = ((size_t)b * p.Hkv + g) * p.n_splits;
  const size_t slot = slot0 + s;
#pragma unroll
  for (int h = 0; h < REP; ++h) p.ws_acc[(slot * REP + h) * kD + tid] = oo[h];
  if (tid < REP) {
    p.ws_ml[(slot * REP + tid) * 2 + 0] = MM[tid];
    p.ws_ml[(slot * REP + tid) * 2 + 1] = LL[tid];
  }
  __syncthreads();
  if (tid == 0)  // release the CTA's writes (ordered by the barrier), acquire the others', one round trip
    s_ticket = atom_add_acq_rel_gpu(p.ws_cnt + (size_t)b * p.Hkv + g, 1);
  __syncthreads();
  if (s_ticket != n_act - 1) return;

  float* sW = (float*)ring + kW * kHP * kD;   // [kMaxSplitsM][REP] weights, then [REP] totals
  float* sLk = sW + kMaxSplitsM * REP;
  float* sTot = sLk + kMaxSplitsM * REP;
  for (int idx = tid; idx < n_act * REP; idx += kTh) {
    sW[idx] = __ldcg(p.ws_ml + (slot0 * REP + idx) * 2);
    sLk[idx] = __ldcg(p.ws_ml + (slot0 * REP + idx) * 2 + 1);
  }
  __syncthreads();
  if (tid < REP) {
    float M = -INFINITY;
    for (int k = 0; k < n_act; ++k) M = fmaxf(M, sW[k * REP + tid]);
    float L = 0.f;
    for (int k = 0; k < n_act; ++k) {
      const float w = sW[k * REP + tid] == -INFINITY ? 0.f : exp2f(sW[k * REP + tid] - M);
      sW[k * REP + tid] = w;
      L = fmaf(w, sLk[k * REP + tid], L);
    }
    sTot[tid] = L;
  }
  __syncthreads();
  float O[REP];
#pragma unroll
  for (int h = 0; h < REP; ++h) O[h] = 0.f;
  const float* accp = p.ws_acc + slot0 * REP * kD + tid;
  constexpr int kU = REP >= 8 ? 8 : 16;  // splits of loads in flight per thread
  for (int k0 = 0; k0 < n_act; k0 += kU) {
    float v[kU][REP];
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (k0 + u < n_act)
#pragma unroll
        for (int h = 0; h < REP; ++h) v[u][h] = __ldcg(accp + ((size_t)(k0 + u) * REP + h) * kD);
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (k0 + u < n_act)
#pragma unroll
        for (int h = 0; h < REP; ++h) O[h] = fmaf(sW[(k0 + u) * REP + h], v[u][h], O[h]);
  }
#pragma unroll
  for (int h = 0; h < REP; ++h) {
    const float r = O[h] / sTot[h];
    if (p.out_bf16) p.out_bf16[(head0 + h) * kD + tid] = __float2bfloat16_rn(r);
    else p.out_f32[(head0 + h) * kD + tid] = r;
  }
  if (tid == 0) p.ws_cnt[(size_t)b * p.Hkv + g] = 0;
}

constexpr size_t smem_bytes(int rep, int kSt) {
  return 1024 + (size_t)kSt * 2 * kTileBytes + 2 * kHP * kD * 2 + (size_t)kW * 2 * kHP * 16 * 2 +
         (size_t)rep * kD * 4 + 2 * kW * kHP * 4 + 4 * 9 * 4 + 64 + (size_t)kSt * kW * 8;
}

// QD_ATTN_TMA=0 keeps the cp.async loads on every page size.
bool tma_enabled() {
  static const bool on = [] {
    const char* v = getenv("QD_ATTN_TMA");
    return v == nullptr || atoi(v) != 0;
  }();
  return on;
}

template <int REP, bool FUSED, int ST>
cudaError_t launch_m(const MParams& p, const Launch& L) {
  // TMA boxes need 16-row page segments; other page sizes take the cp.async form
  alignas(64) CUtensorMap tk, tv;
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  bool tma = p.page_size % 16 == 0 && tma_enabled();
  if (tma) {
    const uint64_t rows = (uint64_t)p.n_pages * p.Hkv * p.page_size;
    tma = encode_tmap_bf16_2d(&tk, p.k_pages, rows, kD, 16) == cudaSuccess &&
          encode_tmap_bf16_2d(&tv, p.v_pages, rows, kD, 16) == cudaSuccess;
  }
  const size_t smem = smem_bytes(REP, ST);
  if (tma) {
    auto k = attn_mma_kernel<REP, FUSED, ST, true>;
    static bool attr_set = false;
    if (!attr_set) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr_set = true;
    }
    return launch_ex(k, dim3(p.n_splits, p.Hkv, p.B), dim3(kTh), smem, L, tk, tv, p);
  }
  auto k = attn_mma_kernel<REP, FUSED, ST, false>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(k, dim3(p.n_splits, p.Hkv, p.B), dim3(kTh), smem, L, tk, tv, p);
}

// 2-stage ring by default: ~74 KB of shared memory leaves room on the SM for
// the next GEMV's CTA, which then prefetches its weights while attention runs.
// QD_ATTN_STAGES=4 keeps a whole 256-token split in flight at small batch.
template <int REP, bool FUSED>
cudaError_t launch_ms(const MParams& p, const Launch& L) {
  static const int deep = [] {
    const char* v = getenv("QD_ATTN_STAGES");
    return v ? atoi(v) : 2;
  }();
  const long long ctas = (long long)p.n_splits * p.Hkv * p.B;
  if (deep >= 4 && ctas <= 2LL * dev_info().sm_count) return launch_m<REP, FUSED, 4>(p, L);
  return launch_m<REP, FUSED, 2>(p, L);
}

}  // namespace

// Same workspace layout as the CUDA-core form: [slots][REP][128] partials,
// [slots][REP][2] (max, sum), [B * Hkv] tickets; chunk is a multiple of 128.
cudaError_t launch_attention_mma(const AttnArgs& a, int chunk, size_t slots, const Launch& L) {
  MParams p = {};
  const int rep = a.Hq / a.Hkv;
  p.q = a.q;
  p.qkv = a.qkv;
  p.q_norm = (const __nv_bfloat16*)a.q_norm;
  p.k_norm = (const __nv_bfloat16*)a.k_norm;
  p.rope = (const float2*)a.rope;
  p.rope_max_pos = a.rope_max_pos;
  p.eps = a.eps;
  p.act_bf16 = a.act_bf16;
  p.pos = a.pos;
  p.seq_lens = a.seq_lens;
  p.k_pages = (const __nv_bfloat16*)a.k_pages;
  p.v_pages = (const __nv_bfloat16*)a.v_pages;
  p.k_pages_w = (__nv_bfloat16*)a.k_pages;
  p.v_pages_w = (__nv_bfloat16*)a.v_pages;
  p.page_table = a.page_table;
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv;
  p.page_size = a.page_size; p.max_pages = a.max_pages; p.n_pages = a.n_pages;
  p.chunk = chunk;
  p.n_splits = (a.max_ctx + chunk - 1) / chunk;
  p.scale_log2 = a.scale * kLog2e;
  p.out_f32 = a.out_f32;
  p.out_bf16 = (__nv_bfloat16*)a.out_bf16;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  unsigned char* ws = (unsigned char*)a.workspace;
  p.ws_acc = (float*)ws;
  p.ws_ml = (float*)(ws + al(slots * rep * kD * 4));
  p.ws_cnt = (int*)(ws + al(slots * rep * kD * 4) + al(slots * rep * 2 * 4));
  p.err = L.err;
  p.trig_late = L.trig_late;
  p.kv_ready = a.kv_ready;
  const bool fused = a.qkv != nullptr;
  switch (rep) {
    case 1: return fused ? launch_ms<1, true>(p, L) : launch_ms<1, false>(p, L);
    case 2: return fused ? launch_ms<2, true>(p, L) : launch_ms<2, false>(p, L);
    case 4: return fused ? launch_ms<4, true>(p, L) : launch_ms<4, false>(p, L);
    case 8: return fused ? launch_ms<8, true>(p, L) : launch_ms<8, false>(p, L);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qd
