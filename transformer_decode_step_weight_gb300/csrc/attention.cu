// GQA split-KV decode attention over a paged bf16 KV cache, with the per-head
// QK RMSNorm, RoPE and the K/V cache write of the current token fused in.
//
// "qwen3-8b-rtx4080-cutedsl" README, "Split-KV decode attention": the sequence
// is split across CTAs (Flash-Decoding) and a final pass combines the partial
// softmax states; the q heads that share a KV head are packed into one CTA.
// Same README, "GQA + QK-Norm": kv head = q head / (Hq / Hkv); per-head RMSNorm
// of q and k before the scores. "GPU Kernel Lab" README, "Decode integration":
// Q/K RMSNorm + RoPE + direct K/V cache write, then split-KV online-softmax
// attention; "Measured final results": K/V in fixed physical pages read
// through a page table.
//
// GB300 design:
//   * grid (split, kv head, sequence), 512 threads (256 for 8 q heads per kv
//     head); a CTA owns `chunk` tokens
//     (a multiple of 128) of one kv head and all REP = Hq/Hkv q heads reading it;
//     the host sizes `chunk` so the grid is about one CTA per SM at batch 1
//     and one split per sequence at large batch;
//   * the chunk streams through shared memory in 64-token tiles: one thread
//     issues TMA bulk copies (cp.async.bulk, one per contiguous page segment)
//     of a tile's K and V rows into a 3-stage ring on mbarriers, the first
//     stages before the programmatic-dependent wait (~100 KB of shared memory,
//     so the CTA fits beside the projection kernel it overlaps);
//   * per tile: scores from shared memory in f32, an online-softmax update of
//     the running (max, sum) per head, then P.V into per-lane accumulators;
//   * a split publishes (m, l, acc[REP][128]) to the workspace and takes a
//     ticket; the last split of a (sequence, kv head) combines all partials in
//     split order (fixed, so results are deterministic) with every load issued
//     in parallel, and resets the ticket. No spin-wait anywhere.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace qd {
namespace {

constexpr int kD = 128;
constexpr int kTile = 64;
// K/V ring depth: 3 stages by default; QD_ATTN_SIMT_STAGES = 2..4 (4 puts a whole
// 256-token split in flight before the dependency wait).
constexpr int kMaxStages = 4;
// 256 threads (8 warps) per CTA, with about two CTAs per SM (attn_chunk): on the
// Qwen3-8B step 338.0 vs 335.3 tok/s against 512 threads and one CTA per SM, on
// Qwen3-0.6B 1447 vs 1281 (same box).
__host__ __device__ constexpr int threads_for(int rep) { return 256; }
constexpr int kMaxSplits = 256;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
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
  __nv_bfloat16* k_pages;
  __nv_bfloat16* v_pages;
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
  L2Prefetch pf[2];
  int pf_late;  // 1: prefetch once this CTA's own K/V tiles have all arrived
  int stages;   // K/V ring depth, 2..kMaxStages
  int trig_loop;  // 1: trigger the dependent launch after the K/V loop, not at the start
  const __nv_bfloat16* k_next;  // the next layer's caches: this split's rows go to L2
  const __nv_bfloat16* v_next;
  int kv_pf;                    // 0 off, 1 evict-normal, 2 evict-last
  int kv_ready;                 // the current token's K/V rows are already in the cache
};

struct Carve {
  size_t kv, q, s, run, wm, bar, total;
};
__host__ __device__ inline Carve carve(int rep, int stages) {
  Carve c;
  c.kv = 0;                                          // stages x (K tile, V tile)
  c.q = c.kv + (size_t)stages * 2 * kTile * kD * 2;
  c.s = c.q + (size_t)rep * kD * 4;                  // per-warp probabilities, REP x 64 floats in all
  c.run = c.s + (size_t)rep * kTile * 4;             // m[REP], l[REP], scratch
  c.wm = c.run + 64 * 4;                             // per-warp maxima / sums [2][16 warps][8]
  c.bar = c.wm + 2 * 16 * 8 * 4;                     // full[kMaxStages], empty[kMaxStages]
  c.total = c.bar + 2 * kMaxStages * 8;
  return c;
}

// N adjacent floats through L2 (partials written by other CTAs of this grid).
template <int N>
QD_DEV void load_cg(const float* src, float* dst) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int j = 0; j < N; j += 4) {
      const float4 v = __ldcg((const float4*)(src + j));
      dst[j] = v.x; dst[j + 1] = v.y; dst[j + 2] = v.z; dst[j + 3] = v.w;
    }
  } else if constexpr (N == 2) {
    const float2 v = __ldcg((const float2*)src);
    dst[0] = v.x; dst[1] = v.y;
  } else {
    dst[0] = __ldcg(src);
  }
}

// Issue the TMA copies of tile rows [t, t + n) of kv head g into stage smem.
QD_DEV void issue_tile(const AttnParams& p, int b, int g, int t, int n, __nv_bfloat16* sK, __nv_bfloat16* sV,
                       uint64_t* bar) {
  mbar_arrive_expect_tx(bar, (uint32_t)n * kD * 2 * 2);
  const int32_t* pt = p.page_table + (size_t)b * p.max_pages;
  const int ps = p.page_size;
  const int t0 = t, end = t + n;
  while (t < end) {
    const PagedSlot ps_t = paged_slot(pt, t, ps, p.n_pages);
    if (!ps_t.ok) set_error(p.err, QD_DEVERR_PAGE);
    const int seg_end = min(end, t + (ps - ps_t.slot));
    const size_t off = (((size_t)ps_t.page * p.Hkv + g) * ps + ps_t.slot) * kD;
    const uint32_t bytes = (uint32_t)(seg_end - t) * kD * 2;
    bulk_g2s(sK + (size_t)(t - t0) * kD, p.k_pages + off, bytes, bar);
    bulk_g2s(sV + (size_t)(t - t0) * kD, p.v_pages + off, bytes, bar);
    t = seg_end;
  }
}

// Fetch cached rows [t0, t1) of kv head g of sequence b of another layer's
// caches (same shape as this layer's) into L2: one page segment per lane.
QD_DEV void prefetch_kv_rows(const AttnParams& p, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int b, int g,
                             int t0, int t1, int lane, uint64_t pol) {
  if (t1 <= t0) return;
  const int ps = p.page_size;
  const int32_t* pt = p.page_table + (size_t)b * p.max_pages;
  for (int lp = t0 / ps + lane; lp <= (t1 - 1) / ps; lp += 32) {
    const int page = pt[lp];
    if (page < 0 || page >= p.n_pages) continue;
    const int a = max(t0, lp * ps), e = min(t1, (lp + 1) * ps);
    const size_t off = (((size_t)page * p.Hkv + g) * ps + (a - lp * ps)) * kD;
    const uint32_t bytes = (uint32_t)(e - a) * kD * 2;
    l2_prefetch_hint(kc + off, bytes, pol);
    l2_prefetch_hint(vc + off, bytes, pol);
  }
}

// Thread-block-cluster helpers: a full cluster barrier and distributed shared
// memory loads from a peer CTA (the cluster spans grid x, so a CTA's rank in
// its cluster is blockIdx.x).
QD_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
QD_DEV float ld_peer(const float* local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

// CLUSTER = false: split s of `chunk` tokens, partials through the workspace and
//   a ticket (the last split combines).
// CLUSTER = true: the gridDim.x CTAs of a (kv head, sequence) form one thread
//   block cluster and split the sequence evenly; the partials stay in shared
//   memory and are combined through distributed shared memory after a cluster
//   barrier (no workspace, no ticket, no global round trip).
template <int REP, bool FUSED, bool CLUSTER>
__global__ void __launch_bounds__(threads_for(REP)) attn_kernel(const AttnParams p) {
  constexpr int kThreads = threads_for(REP);
  constexpr int kWarps = kThreads / 32;
  constexpr int kPairs = kTile / 2 / kWarps;  // token pairs per warp per tile
  extern __shared__ __align__(128) unsigned char smem[];
  const int kStages = p.stages;
  const Carve cv = carve(REP, kStages);
  __nv_bfloat16* sKV = (__nv_bfloat16*)(smem + cv.kv);
  float* sQ = (float*)(smem + cv.q);
  float* sS = (float*)(smem + cv.s);
  float* sRun = (float*)(smem + cv.run);  // [0,REP) m, [8,8+REP) l, [16,16+REP) alpha, [32,36) scratch
  uint64_t* bars = (uint64_t*)(smem + cv.bar);
  __shared__ int s_ticket;
  __shared__ float s_x[kD];

  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // DRAM is mostly idle while this short kernel runs: every CTA fetches its share
  // of the next GEMVs' weights into L2 once the dependency wait is over (the
  // projection before this kernel is complete then, so it loses no bandwidth).
  auto prefetch_next = [&]() {
    if (warp == 1) {
      const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
      const unsigned n_cta = gridDim.x * gridDim.y * gridDim.z;
      l2_prefetch_spans(p.pf[0], cta, n_cta, lane);
      l2_prefetch_spans(p.pf[1], cta, n_cta, lane);
    }
  };

  // The position, the page table and the cached K/V rows below `pos` are not
  // written by the kernel this one waits on (the QKV projection): `pos` was
  // last written by the previous step's argmax, and the cache rows by earlier
  // steps, all complete before the QKV projection's CTAs started. So the first
  // tiles are requested before the programmatic-dependent wait, and stream in
  // while the projection finishes; only q/k/v need the wait.
  if (!p.trig_late && !p.trig_loop) pdl_launch_dependents();

  int len, pos = 0;
  if (FUSED) {
    pos = p.pos[b];
    len = pos + 1;
  } else {
    len = p.seq_lens[b];
  }
  const int cap = p.max_pages * p.page_size;
  if (len < 0 || len > cap || (FUSED && (pos < 0 || pos >= p.rope_max_pos))) {
    if (s == 0 && tid == 0) set_error(p.err, QD_DEVERR_POS);
    pdl_launch_dependents();
    return;
  }
  const size_t head0 = (size_t)b * p.Hq + g * REP;
  if (!CLUSTER && len == 0) {  // empty sequence (standalone form only): zero output
    if (s == 0 && !FUSED)
      for (int e = tid; e < REP * kD; e += kThreads) p.out_f32[head0 * kD + e] = 0.f;
    return;
  }
  int n_act = 1, t0, t_end;                          // keys [t0, t_end)
  if (CLUSTER) {
    const long long cl = gridDim.x;
    t0 = (int)(((long long)len * s) / cl);
    t_end = (int)(((long long)len * (s + 1)) / cl);
  } else {
    n_act = (len + p.chunk - 1) / p.chunk;
    if (s >= n_act) {  // no keys for this split: only its share of the prefetch
      pdl_wait();
      prefetch_next();
      return;
    }
    t0 = s * p.chunk;
    t_end = min(t0 + p.chunk, len);
  }
  const int n_tiles = (t_end - t0 + kTile - 1) / kTile;
  // in the fused form the current token `pos` is not read from the cache
  const int copy_end = (FUSED && !p.kv_ready) ? min(t_end, pos) : t_end;

  auto stage_k = [&](int st) { return sKV + (size_t)st * 2 * kTile * kD; };
  auto stage_v = [&](int st) { return sKV + (size_t)st * 2 * kTile * kD + kTile * kD; };

  uint64_t* empty = bars + kMaxStages;  // a stage is free once every warp has read it
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&bars[st], 1);
      mbar_init(&empty[st], kWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int st = 0; st < kStages && st < n_tiles; ++st) {
      const int ts = t0 + st * kTile;
      issue_tile(p, b, g, ts, max(0, min(ts + kTile, copy_end) - ts), stage_k(st), stage_v(st), &bars[st]);
    }
  }
  // The RoPE row, the QK-norm weights and the cache page of the current token
  // do not come from the previous kernel either: load them before the wait.
  float k_new = 0.f, v_new = 0.f;
  const bool own_pos = FUSED && !p.kv_ready && pos >= t0 && pos < t_end;
  const int d = tid & (kD - 1);
  float2 cs = make_float2(0.f, 0.f);
  float wq = 0.f, wk = 0.f;
  PagedSlot own = {0, 0, false};
  if (FUSED) {
    cs = p.rope[(size_t)pos * (kD / 2) + (d & 63)];
    wq = __bfloat162float(p.q_norm[d]);
    wk = __bfloat162float(p.k_norm[d]);
    if (own_pos) own = paged_slot(p.page_table + (size_t)b * p.max_pages, pos, p.page_size, p.n_pages);
  }
  pdl_wait();  // q, k, v (and, standalone, the caller's q) come from the previous kernel
  if (!p.pf_late) prefetch_next();

  // ---- q for the REP heads of this kv head (pre-scaled by scale * log2 e); new k, v.
  // All head vectors load at once; one barrier for the sums of squares, one for RoPE.
  if (FUSED) {
    const int qkv_w = (p.Hq + 2 * p.Hkv) * kD;
    const float* qkv = p.qkv + (size_t)b * qkv_w;
    // threads [0, 128) own one dim of every head vector; the rest only join the barriers
    const bool dim_thread = tid < kD;
    float xv[REP + 1];
#pragma unroll
    for (int i = 0; i < REP; ++i) xv[i] = dim_thread ? qkv[(g * REP + i) * kD + d] : 0.f;
    xv[REP] = (own_pos && dim_thread) ? qkv[(p.Hq + g) * kD + d] : 0.f;
    const float vx = (own_pos && dim_thread) ? qkv[(p.Hq + p.Hkv + g) * kD + d] : 0.f;
    float* red = sS;  // [4 warps][REP + 1] scratch before the first tile
#pragma unroll
    for (int i = 0; i <= REP; ++i) {
      const float ss = warp_sum(xv[i] * xv[i]);
      if (lane == 0 && dim_thread) red[warp * (REP + 1) + i] = ss;
    }
    __syncthreads();
    float y[REP + 1];
#pragma unroll
    for (int i = 0; i <= REP; ++i) {
      const float tot = (red[i] + red[(REP + 1) + i]) + (red[2 * (REP + 1) + i] + red[3 * (REP + 1) + i]);
      const float inv = 1.0f / sqrtf(tot / (float)kD + p.eps);
      float n = xv[i] * inv;
      if (p.act_bf16) n = round_bf16(n);
      y[i] = (i < REP ? wq : wk) * n;
      if (p.act_bf16) y[i] = round_bf16(y[i]);
      if (dim_thread) {
        if (i < REP) sQ[i * kD + d] = y[i];
        else s_x[d] = y[i];
      }
    }
    __syncthreads();
    float r[REP + 1];
#pragma unroll
    for (int i = 0; i <= REP; ++i) {
      const float other = i < REP ? sQ[i * kD + (d ^ 64)] : s_x[d ^ 64];
      r[i] = (d < 64) ? (y[i] * cs.x - other * cs.y) : (y[i] * cs.x + other * cs.y);
    }
    __syncthreads();
    if (dim_thread) {
#pragma unroll
      for (int i = 0; i < REP; ++i) sQ[i * kD + d] = r[i] * p.scale_log2;
    }
    if (own_pos && dim_thread) {  // this split holds the current token: store k, v in the cache
      k_new = round_bf16(r[REP]);
      v_new = round_bf16(vx);
      if (!own.ok) {
        if (tid == 0) set_error(p.err, QD_DEVERR_PAGE);
      } else {
        const size_t off = (((size_t)own.page * p.Hkv + g) * p.page_size + own.slot) * kD + d;
        p.k_pages[off] = __float2bfloat16_rn(k_new);
        p.v_pages[off] = __float2bfloat16_rn(v_new);
      }
    }
  } else {
    for (int e = tid; e < REP * kD; e += kThreads) sQ[e] = p.q[head0 * kD + e] * p.scale_log2;
  }
  __syncthreads();

  // ---- K/V loop. Each warp owns kPairs token pairs of every tile from score to
  // P.V: lane = (token of a pair, 16-byte chunk of the head dim). Per tile one
  // CTA barrier publishes the per-warp maxima; every warp then forms the same
  // running max per head and rescales only its own accumulators and partial
  // sums. A stage is handed back through its `empty` barrier (one arrival per
  // warp), so no second CTA barrier is needed per tile.
  const int half = lane >> 4, dc = lane & 15;
  float qr[REP][8];
#pragma unroll
  for (int i = 0; i < REP; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) qr[i][e] = sQ[i * kD + dc * 8 + e];
  float acc[REP][8];
#pragma unroll
  for (int i = 0; i < REP; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
  float m_run[REP];                      // identical in every lane of every warp
#pragma unroll
  for (int i = 0; i < REP; ++i) m_run[i] = -INFINITY;
  float l_hold = 0.f;                    // holder lanes: sum of p of head hsel over this lane's tokens
  constexpr int kTokW = 2 * kPairs;      // tokens per warp per tile
  float* sP = sS + warp * REP * kTokW;   // this warp's probabilities [REP][kTokW]
  float* sWm = (float*)(smem + cv.wm);   // [2][16][8]
  constexpr int kHoldMask = 16 / REP - 1;
  const bool holder = (dc & kHoldMask) == 0;
  // head whose dot a holder lane ends with (fixed by the lane's position in the butterfly)
  int hsel = 0;
#pragma unroll
  for (int L = 8, n = REP; L >= 1 && n > 1; L >>= 1) {
    n /= 2;
    if (lane & L) hsel += n;
  }

  for (int it = 0; it < n_tiles; ++it) {
    const int st = it % kStages;
    const int ts = t0 + it * kTile;
    const int nv = min(kTile, t_end - ts);
    __nv_bfloat16* sK = stage_k(st);
    __nv_bfloat16* sV = stage_v(st);
    const bool got = mbar_wait_bounded(&bars[st], (uint32_t)((it / kStages) & 1), p.err);
    if (own_pos && pos >= ts && pos < ts + kTile) {  // CTA-uniform: the current token's row
      if (tid < kD) {
        sK[(size_t)(pos - ts) * kD + tid] = __float2bfloat16_rn(k_new);
        sV[(size_t)(pos - ts) * kD + tid] = __float2bfloat16_rn(v_new);
      }
      __syncthreads();
    }

    // scores of this warp's tokens; after the transposed butterfly over the 16
    // lanes of a token, holder lane (dc) has the full dot of head hsel
    float sc[kPairs];
#pragma unroll
    for (int q = 0; q < kPairs; ++q) {
      const int tt = 2 * (warp * kPairs + q) + half;
      const bool ok = tt < nv;
      uint4 kw = make_uint4(0u, 0u, 0u, 0u);
      if (ok) kw = *(const uint4*)(sK + (size_t)tt * kD + dc * 8);
      const float kf[8] = {bf_lo(kw.x), bf_hi(kw.x), bf_lo(kw.y), bf_hi(kw.y),
                           bf_lo(kw.z), bf_hi(kw.z), bf_lo(kw.w), bf_hi(kw.w)};
      float v[REP];
#pragma unroll
      for (int i = 0; i < REP; ++i) {
        float a = 0.f, c = 0.f;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          a = fmaf(kf[e], qr[i][e], a);
          c = fmaf(kf[e + 1], qr[i][e + 1], c);
        }
        v[i] = a + c;
      }
#pragma unroll
      for (int L = 8, n = REP; L >= 1; L >>= 1) {
        if (n > 1) {
          const int h = n / 2;
          const bool up = (lane & L) != 0;
#pragma unroll
          for (int k = 0; k < h; ++k) {
            const float send = up ? v[k] : v[k + h];
            const float keep = up ? v[k + h] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, L);
          }
          n = h;
        } else {
          v[0] += __shfl_xor_sync(0xffffffffu, v[0], L);
        }
      }
      sc[q] = ok ? v[0] : -INFINITY;
    }
    // this warp's maximum per head -> shared memory (buffer it & 1)
    float mx = sc[0];
#pragma unroll
    for (int q = 1; q < kPairs; ++q) mx = fmaxf(mx, sc[q]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    float* wmb = sWm + (it & 1) * 16 * 8;
    if (holder && half == 0) wmb[warp * 8 + hsel] = mx;
    if (!__syncthreads_and(got)) {  // a K/V copy never arrived: drain, leave together
      for (int k = 1; k < kStages && it + k < n_tiles; ++k)
        mbar_wait_bounded(&bars[(it + k) % kStages], (uint32_t)(((it + k) / kStages) & 1), p.err);
      if (!CLUSTER) return;
      break;  // cluster peers still expect this CTA at the cluster barriers (the error word is set)
    }
    // running max over all warps: lane j < REP reduces head j, then broadcast
    float mh = -INFINITY;
    if (lane < REP) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) mh = fmaxf(mh, wmb[w * 8 + lane]);
    }
    float alpha[REP];
#pragma unroll
    for (int i = 0; i < REP; ++i) {
      const float m_new = fmaxf(m_run[i], __shfl_sync(0xffffffffu, mh, i));
      alpha[i] = exp2f(m_run[i] - m_new);   // 0 on the first tile
      m_run[i] = m_new;
    }
    // probabilities of this warp's tokens (holder lanes), partial sums, P.V
    float m_h = m_run[0], a_h = alpha[0];
#pragma unroll
    for (int i = 1; i < REP; ++i)
      if (hsel == i) { m_h = m_run[i]; a_h = alpha[i]; }
    l_hold *= a_h;
#pragma unroll
    for (int q = 0; q < kPairs; ++q) {
      const float pp = exp2f(sc[q] - m_h);   // 0 for masked tokens
      if (holder) {
        l_hold += pp;
        sP[hsel * kTokW + 2 * q + half] = pp;
      }
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < REP; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[i][e] *= alpha[i];
#pragma unroll
    for (int q = 0; q < kPairs; ++q) {
      const int tt = 2 * (warp * kPairs + q) + half;
      if (tt < nv) {
        const uint4 vw = *(const uint4*)(sV + (size_t)tt * kD + dc * 8);
        const float vf[8] = {bf_lo(vw.x), bf_hi(vw.x), bf_lo(vw.y), bf_hi(vw.y),
                             bf_lo(vw.z), bf_hi(vw.z), bf_lo(vw.w), bf_hi(vw.w)};
#pragma unroll
        for (int i = 0; i < REP; ++i) {
          const float pp = sP[i * kTokW + 2 * q + half];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(pp, vf[e], acc[i][e]);
        }
      }
    }
    __syncwarp();                          // this warp is done with the stage and sP
    if (lane == 0) mbar_arrive(&empty[st]);
    if (tid == 0 && it + kStages < n_tiles) {
      if (mbar_wait_bounded(&empty[st], (uint32_t)((it / kStages) & 1), p.err)) {
        const int tn = t0 + (it + kStages) * kTile;
        issue_tile(p, b, g, tn, max(0, min(tn + kTile, copy_end) - tn), sK, sV, &bars[st]);
      }
    }
  }
  // per-head totals: m (same everywhere) and l summed over holder lanes and warps
  {
    float lw = l_hold + __shfl_xor_sync(0xffffffffu, l_hold, 16);
    float* wl = sWm + (n_tiles & 1) * 16 * 8;   // the buffer no warp can still be reading
    if (holder && half == 0) wl[warp * 8 + hsel] = lw;
    __syncthreads();
    if (tid < REP) {
      float L = 0.f;
      for (int w = 0; w < kWarps; ++w) L += wl[w * 8 + tid];
      float m = m_run[0];
#pragma unroll
      for (int i = 1; i < REP; ++i)
        if (tid == i) m = m_run[i];
      sRun[tid] = m;
      sRun[8 + tid] = L;
    }
  }

  pdl_launch_dependents();  // all K/V of this split is in shared memory
  if (p.pf_late) prefetch_next();
  // DRAM idles while the splits publish and combine: bring the next layer's
  // rows of this split into L2 for its attention
  if (p.kv_pf && p.k_next && warp == 2)
    prefetch_kv_rows(p, p.k_next, p.v_next, b, g, t0, copy_end, lane,
                     p.kv_pf == 2 ? policy_evict_last() : policy_evict_normal());

  // ---- reduce the two token halves, then the warps, element by element
#pragma unroll
  for (int i = 0; i < REP; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] += __shfl_xor_sync(0xffffffffu, acc[i][e], 16);
  constexpr int NE = REP * kD;          // elements of the [REP][128] output
  float* sRed = (float*)sKV;            // [kWarps][REP][128] f32 (the ring is idle now)
  if (half == 0) {
#pragma unroll
    for (int i = 0; i < REP; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) sRed[warp * NE + i * kD + dc * 8 + e] = acc[i][e];
  }
  __syncthreads();
  constexpr int kEpt = NE >= kThreads ? NE / kThreads : 1;   // elements per thread
  const int e0 = tid * kEpt;             // this thread's elements [e0, e0 + kEpt) (one head)
  const bool elem_thread = e0 < NE;
  const int hi = elem_thread ? e0 / kD : 0;
  float o[kEpt];
#pragma unroll
  for (int j = 0; j < kEpt; ++j) {
    float a = 0.f;
    if (elem_thread) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) a += sRed[w * NE + e0 + j];
    }
    o[j] = a;
  }

  if (CLUSTER && gridDim.x > 1) {
    float* sPart = sRed + kWarps * NE;   // this CTA's unnormalised partial [NE]
    if (elem_thread) {
#pragma unroll
      for (int j = 0; j < kEpt; ++j) sPart[e0 + j] = o[j];
    }
    cluster_sync();  // every CTA's (m, l, partial) is visible cluster-wide
    const uint32_t cl = gridDim.x;
    const int per = NE / (int)cl;        // output elements combined by this CTA
    for (int e = tid; e < per; e += kThreads) {
      const int el = s * per + e, i = el / kD;
      float M = -INFINITY;
      for (uint32_t r = 0; r < cl; ++r) M = fmaxf(M, ld_peer(&sRun[i], r));
      float L = 0.f, O = 0.f;
      for (uint32_t r = 0; r < cl; ++r) {
        const float w = exp2f(ld_peer(&sRun[i], r) - M);
        L = fmaf(w, ld_peer(&sRun[8 + i], r), L);
        O = fmaf(w, ld_peer(&sPart[el], r), O);
      }
      const float res = O / L;
      if (p.out_bf16) p.out_bf16[head0 * kD + el] = __float2bfloat16_rn(res);
      else p.out_f32[head0 * kD + el] = res;
    }
    cluster_sync();  // peers may still be reading this CTA's shared memory
    return;
  }

  if (n_act == 1) {  // one split (or a cluster of one): already complete
    if (elem_thread) {
      const float inv = 1.0f / sRun[8 + hi];
#pragma unroll
      for (int j = 0; j < kEpt; ++j) {
        const float r = o[j] * inv;
        if (p.out_bf16) p.out_bf16[head0 * kD + e0 + j] = __float2bfloat16_rn(r);
        else p.out_f32[head0 * kD + e0 + j] = r;
      }
    }
    return;
  }

  // ---- publish the partial, take a ticket; the last split combines
  const size_t slot0 = ((size_t)b * p.Hkv + g) * p.n_splits;
  const size_t slot = slot0 + s;
  if (elem_thread) {
#pragma unroll
    for (int j = 0; j < kEpt; ++j) p.ws_acc[slot * NE + e0 + j] = o[j];
  }
  if (tid < REP) {
    p.ws_ml[(slot * REP + tid) * 2 + 0] = sRun[tid];
    p.ws_ml[(slot * REP + tid) * 2 + 1] = sRun[8 + tid];
  }
  __syncthreads();  // every thread's share of the partial is written
  if (tid == 0)     // release the CTA's writes, take a ticket, acquire the others' (one round trip)
    s_ticket = atom_add_acq_rel_gpu(p.ws_cnt + (size_t)b * p.Hkv + g, 1);
  __syncthreads();
  if (s_ticket != n_act - 1) return;

  // The last split combines. One round of L2 loads: this thread's elements of the
  // first kB splits' partials go to registers while (m, l) of every split go to
  // shared memory; weights w[k][i] = exp2(m_k - M_i) and totals L_i follow.
  constexpr int kB = 32 / kEpt > 0 ? 32 / kEpt : 1;   // splits per batch of register loads
  float* sW = (float*)sKV + kWarps * NE;        // after sRed: [kMaxSplits][REP]
  float* sLk = sW + kMaxSplits * REP;           // [kMaxSplits][REP]
  float* sL = sLk + kMaxSplits * REP;           // [REP]
  const float* accp = p.ws_acc + slot0 * NE + e0;
  float v[kB][kEpt];
  if (elem_thread) {
#pragma unroll
    for (int u = 0; u < kB; ++u)
      if (u < n_act) load_cg<kEpt>(accp + (size_t)u * NE, v[u]);
  }
  for (int idx = tid; idx < n_act * REP; idx += kThreads) {
    const float2 ml = __ldcg((const float2*)(p.ws_ml + (slot0 * REP + idx) * 2));
    sW[idx] = ml.x;
    sLk[idx] = ml.y;
  }
  __syncthreads();
  if (tid < REP) {
    float M = -INFINITY;
    for (int k = 0; k < n_act; ++k) M = fmaxf(M, sW[k * REP + tid]);
    float L = 0.f;
    for (int k = 0; k < n_act; ++k) {
      const float w = exp2f(sW[k * REP + tid] - M);
      sW[k * REP + tid] = w;
      L = fmaf(w, sLk[k * REP + tid], L);
    }
    sL[tid] = L;
  }
  __syncthreads();
  if (elem_thread) {
    float O[kEpt];
#pragma unroll
    for (int j = 0; j < kEpt; ++j) O[j] = 0.f;
    for (int k0 = 0; k0 < n_act; k0 += kB) {
      if (k0 > 0) {
#pragma unroll
        for (int u = 0; u < kB; ++u)
          if (k0 + u < n_act) load_cg<kEpt>(accp + (size_t)(k0 + u) * NE, v[u]);
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        if (k0 + u < n_act) {
          const float w = sW[(k0 + u) * REP + hi];
#pragma unroll
          for (int j = 0; j < kEpt; ++j) O[j] = fmaf(w, v[u][j], O[j]);
        }
      }
    }
    const float invL = 1.0f / sL[hi];
#pragma unroll
    for (int j = 0; j < kEpt; ++j) {
      const float r = O[j] * invL;
      if (p.out_bf16) p.out_bf16[head0 * kD + e0 + j] = __float2bfloat16_rn(r);
      else p.out_f32[head0 * kD + e0 + j] = r;
    }
  }
  if (tid == 0) p.ws_cnt[(size_t)b * p.Hkv + g] = 0;
}

__global__ void rope_table_kernel(float2* table, int max_pos, int half, double theta) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)max_pos * half) return;
  const int p = (int)(i / half), j = (int)(i % half);
  const double inv = pow(theta, -2.0 * (double)j / (double)(2 * half));
  double sn, cs;
  sincos((double)p * inv, &sn, &cs);
  table[i] = make_float2((float)cs, (float)sn);
}

template <int REP, bool FUSED, bool CLUSTER>
cudaError_t launch_rep(const AttnParams& prm, int cluster, const Launch& L) {
  auto k = attn_kernel<REP, FUSED, CLUSTER>;
  const size_t smem = carve(REP, prm.stages).total;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)carve(REP, kMaxStages).total);
    if (e != cudaSuccess) return e;
    if (CLUSTER) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    attr_set = true;
  }
  if (CLUSTER) {
    dim3 grid(cluster, prm.Hkv, prm.B);
    return launch_ex_cluster(k, grid, dim3(threads_for(REP)), smem, cluster, L, prm);
  }
  dim3 grid(prm.n_splits, prm.Hkv, prm.B);
  return launch_ex(k, grid, dim3(threads_for(REP)), smem, L, prm);
}

int simt_stages() {
  static const int n = [] {
    const char* v = getenv("QD_ATTN_SIMT_STAGES");
    return v ? std::max(2, std::min(kMaxStages, atoi(v))) : 3;
  }();
  return n;
}

// Cluster size for the fused step: the smallest power of two that gives about
// one CTA per SM over batch x kv heads, at most 16 (8 if the device cannot
// co-schedule clusters of 16 of this kernel).
template <int REP, bool FUSED>
int pick_cluster(int B, int Hkv, int max_cl) {
  const int sms = dev_info().sm_count;
  const int pairs = std::max(1, B * Hkv);
  int cl = 1;
  while (cl < std::min(16, max_cl) && pairs * cl * 2 <= sms) cl *= 2;
  static int max_ok = 0;
  if (max_ok == 0) {
    auto k = attn_kernel<REP, FUSED, true>;
    max_ok = 8;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)carve(REP, kMaxStages).total) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16, 1, 1);
      cfg.blockDim = dim3(threads_for(REP));
      cfg.dynamicSmemBytes = carve(REP, simt_stages()).total;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 16;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess && n >= 1) max_ok = 16;
    }
    cudaGetLastError();
  }
  return std::min(cl, max_ok);
}

}  // namespace

// Tokens per split: about two CTAs per SM at small batch (256-thread CTAs, two fit
// on an SM; fewer partials for the combine than more splits would give), a single
// split per sequence once batch x kv heads fills the GPU twice, never more than
// kMaxSplits.
int attn_chunk(int B, int Hkv, int max_ctx) {
  const int sms = dev_info().sm_count;
  const int pairs = std::max(1, B * Hkv);
  const int want = std::max(1, (2 * sms + pairs - 1) / pairs);
  int chunk = (max_ctx + want - 1) / want;
  chunk = std::max(kTile, ((chunk + kTile - 1) / kTile) * kTile);
  while ((max_ctx + chunk - 1) / chunk > kMaxSplits) chunk += kTile;
  return chunk;
}

// Sized for the largest split count any device could choose (64-token chunks,
// capped at kMaxSplits), so the size does not depend on the SM count.
static size_t slots_cap(int B, int Hkv, int max_ctx) {
  return (size_t)B * Hkv * std::min<size_t>((size_t)kMaxSplits, (size_t)(max_ctx + kTile - 1) / kTile);
}

size_t attn_workspace_bytes(int B, int Hq, int Hkv, int max_ctx) {
  const int rep = Hq / Hkv;
  const size_t slots = slots_cap(B, Hkv, max_ctx);
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al(slots * rep * kD * 4) + al(slots * rep * 2 * 4) + al((size_t)B * Hkv * 4);
}

// Kernel choice. When batch x kv heads fills the GPU (many CTAs, throughput-
// bound) the tensor-core kernel of attention_mma.cu is used; when there are
// only a few splits per SM (batch 1, latency-bound) the 512-thread CUDA-core
// kernel of this file measured faster (Qwen3-8B step: 301 vs 285-291 tok/s;
// 64 sequences: 3019 vs 4226 tok/s the other way round). QD_ATTN_IMPL=simt|mma
// forces one. Same workspace; results agree within f32 rounding.
static int attn_impl_forced() {
  static const int v = [] {
    const char* e = getenv("QD_ATTN_IMPL");
    if (e && strcmp(e, "simt") == 0) return 1;
    if (e && strcmp(e, "mma") == 0) return 2;
    return 0;
  }();
  return v;
}

// Tokens per split of the tensor-core form (batch x kv heads fill the GPU): short
// splits so that sequences of very different lengths still end together
// (QD_ATTN_MMA_CHUNK, a multiple of 64; default 1024: on 64 sequences of 128 to
// 4096 tokens, 1024 measured faster than 256, 512 and whole sequences).
static int attn_chunk_mma(int max_ctx) {
  static const int forced = [] {
    const char* v = getenv("QD_ATTN_MMA_CHUNK");
    return v ? atoi(v) : 1024;
  }();
  int chunk = std::max(kTile, (forced / kTile) * kTile);
  while ((max_ctx + chunk - 1) / chunk > kMaxSplits) chunk += kTile;
  return chunk;
}

// Tensor-core form below the SM count (from 32 pairs, or forced by QD_ATTN_IMPL=mma):
// the CUDA-core form's split, or QD_ATTN_MMA_SMALL_CHUNK tokens (a multiple of 64).
static int attn_chunk_mma_small(const AttnArgs& a) {
  static const int forced = [] {
    const char* v = getenv("QD_ATTN_MMA_SMALL_CHUNK");
    return v ? atoi(v) : 0;
  }();
  if (forced <= 0) return attn_chunk(a.B, a.Hkv, a.max_ctx);
  int chunk = std::max(kTile, (forced / kTile) * kTile);
  while ((a.max_ctx + chunk - 1) / chunk > kMaxSplits) chunk += kTile;
  return chunk;
}

static bool attn_use_mma(const AttnArgs& a) {
  const int f = attn_impl_forced();
  if (f) return f == 2;
  // From 32 (sequence, kv head) pairs the tensor-core form, with the CUDA-core form's
  // split sizing below the SM count: on the Qwen3-8B step 2058 vs 1819 tok/s at 8
  // sequences, 1153 vs 1144 at 4, equal at 2 (and slower at batch 1).
  return (long long)a.B * a.Hkv >= 32;
}

cudaError_t launch_attention(const AttnArgs& a, const Launch& L) {
  if (attn_use_mma(a) && !(a.qkv && a.use_cluster > 1))
    return launch_attention_mma(a,
                                (long long)a.B * a.Hkv >= dev_info().sm_count ? attn_chunk_mma(a.max_ctx)
                                                                               : attn_chunk_mma_small(a),
                                slots_cap(a.B, a.Hkv, a.max_ctx), L);
  AttnParams p = {};
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
  p.k_pages = (__nv_bfloat16*)a.k_pages;
  p.v_pages = (__nv_bfloat16*)a.v_pages;
  p.page_table = a.page_table;
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv;
  p.page_size = a.page_size; p.max_pages = a.max_pages; p.n_pages = a.n_pages;
  p.chunk = attn_chunk(a.B, a.Hkv, a.max_ctx);
  p.n_splits = (a.max_ctx + p.chunk - 1) / p.chunk;
  p.scale_log2 = a.scale * kLog2e;
  p.out_f32 = a.out_f32;
  p.out_bf16 = (__nv_bfloat16*)a.out_bf16;
  const size_t slots = slots_cap(a.B, a.Hkv, a.max_ctx);
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  unsigned char* ws = (unsigned char*)a.workspace;
  p.ws_acc = (float*)ws;
  p.ws_ml = (float*)(ws + al(slots * rep * kD * 4));
  p.ws_cnt = (int*)(ws + al(slots * rep * kD * 4) + al(slots * rep * 2 * 4));
  p.err = L.err;
  p.trig_late = L.trig_late;
  p.pf[0] = a.pf[0];
  p.pf[1] = a.pf[1];
  p.pf_late = a.pf_late;
  p.stages = simt_stages();
  p.trig_loop = a.trig_loop;
  p.k_next = (const __nv_bfloat16*)a.k_next;
  p.v_next = (const __nv_bfloat16*)a.v_next;
  p.kv_pf = a.kv_pf;
  p.kv_ready = a.kv_ready;
  const bool fused = a.qkv != nullptr;
  // the fused decode step splits each sequence across one thread block cluster;
  // the standalone call keeps the workspace split (its workspace is the scratch)
#define QD_ATTN_CASE(R)                                                                   \
  case R:                                                                                 \
    if (fused && a.use_cluster > 1) return launch_rep<R, true, true>(p, pick_cluster<R, true>(a.B, a.Hkv, a.use_cluster), L); \
    return fused ? launch_rep<R, true, false>(p, 0, L) : launch_rep<R, false, false>(p, 0, L);
  switch (rep) {
    QD_ATTN_CASE(1)
    QD_ATTN_CASE(2)
    QD_ATTN_CASE(4)
    QD_ATTN_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef QD_ATTN_CASE
}

// One CTA of 128 threads per (kv head, row): the k head of the row normed and
// rotated as in the fused prologue above (warp sums combined as (w0 + w1) + (w2 + w3)),
// v as is, both rounded to bf16 and stored at the row's position.
__global__ void __launch_bounds__(kD) kv_write_kernel(const float* qkv, int Hq, int Hkv, const __nv_bfloat16* k_norm,
                                                      const float2* rope, int rope_max_pos, float eps, int act_bf16,
                                                      const int32_t* pos, const int32_t* page_table, int pt_stride,
                                                      int page_size, int max_pages, int n_pages, __nv_bfloat16* k_pages,
                                                      __nv_bfloat16* v_pages, int* err) {
  __shared__ float red[4];
  __shared__ float s_y[kD];
  const int g = blockIdx.x, b = blockIdx.y, d = threadIdx.x, lane = d & 31, warp = d >> 5;
  pdl_wait();
  pdl_launch_dependents();
  const int ps_ = pos[b];
  if (ps_ < 0 || ps_ >= max_pages * page_size || ps_ >= rope_max_pos) {
    if (d == 0) set_error(err, QD_DEVERR_POS);
    return;
  }
  const int qkv_w = (Hq + 2 * Hkv) * kD;
  const float x = qkv[(size_t)b * qkv_w + (Hq + g) * kD + d];
  const float vx = qkv[(size_t)b * qkv_w + (Hq + Hkv + g) * kD + d];
  const float ss = warp_sum(x * x);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  const float tot = (red[0] + red[1]) + (red[2] + red[3]);
  const float inv = 1.0f / sqrtf(tot / (float)kD + eps);
  float n = x * inv;
  if (act_bf16) n = round_bf16(n);
  float y = __bfloat162float(k_norm[d]) * n;
  if (act_bf16) y = round_bf16(y);
  s_y[d] = y;
  __syncthreads();
  const float2 cs = rope[(size_t)ps_ * (kD / 2) + (d & 63)];
  const float other = s_y[d ^ 64];
  const float r = (d < 64) ? (y * cs.x - other * cs.y) : (y * cs.x + other * cs.y);
  const PagedSlot sl = paged_slot(page_table + (size_t)b * pt_stride, ps_, page_size, n_pages);
  if (!sl.ok) {
    if (d == 0) set_error(err, QD_DEVERR_PAGE);
    return;
  }
  const size_t off = (((size_t)sl.page * Hkv + g) * page_size + sl.slot) * kD + d;
  k_pages[off] = __float2bfloat16_rn(round_bf16(r));
  v_pages[off] = __float2bfloat16_rn(round_bf16(vx));
}

cudaError_t launch_kv_write(const float* qkv, int B, int Hq, int Hkv, const void* k_norm, const float* rope,
                            int rope_max_pos, float eps, int act_bf16, const int32_t* pos, const int32_t* page_table,
                            int pt_stride, int page_size, int max_pages, int n_pages, void* k_pages, void* v_pages,
                            const Launch& L) {
  return launch_ex(kv_write_kernel, dim3(Hkv, B), dim3(kD), 0, L, qkv, Hq, Hkv, (const __nv_bfloat16*)k_norm,
                   (const float2*)rope, rope_max_pos, eps, act_bf16, pos, page_table, pt_stride, page_size, max_pages,
                   n_pages, (__nv_bfloat16*)k_pages, (__nv_bfloat16*)v_pages, L.err);
}

cudaError_t launch_rope_table(float* table, int max_pos, int head_dim, float theta, cudaStream_t s) {
  const int half = head_dim / 2;
  const long long n = (long long)max_pos * half;
  const int threads = 256;
  const int blocks = (int)((n + threads - 1) / threads);
  rope_table_kernel<<<blocks, threads, 0, s>>>((float2*)table, max_pos, half, (double)theta);
  return cudaGetLastError();
}

}  // namespace qd

// ---------------------------------------------------------------------------
// Allocation-free form of qd_attn_decode_paged.
//
// Some callers cannot allocate device memory for the split-KV scratch: hosts
// whose device memory is fully reserved up front by their own pool, plugins
// that are handed only input and output buffers, and latency-critical loops
// where cudaMalloc / cudaFree would add an implicit device synchronisation.
// For them the scratch lives in this file-scope device array. Every GPU that
// loads the library holds it until the process exits.
static constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

namespace qd {
namespace {

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of g_attn_scratch on the current device, looked up once per
// device (the name is only a host-side stand-in for the device array).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace qd

namespace qd {

size_t attn_noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

// The ticket counters are the last block of the workspace (see
// attn_workspace_bytes). They must start at zero, and a call that was cut short
// could have left them non-zero, so they are cleared on every call.
cudaError_t attn_noalloc_scratch(int B, int Hq, int Hkv, int max_ctx, void** ptr, cudaStream_t stream) {
  const size_t bytes = attn_workspace_bytes(B, Hq, Hkv, max_ctx);
  const size_t cnt = (((size_t)B * Hkv * 4) + 255) & ~(size_t)255;
  if (bytes > kNoAllocScratchBytes || bytes < cnt) return cudaErrorInvalidValue;
  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync((unsigned char*)base + bytes - cnt, 0, cnt, stream);
  if (e != cudaSuccess) return e;
  *ptr = base;
  return cudaSuccess;
}

}  // namespace qd
