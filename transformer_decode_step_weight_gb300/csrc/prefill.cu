// Prefill of one sequence: the prompt's n tokens through a layer at once, with
// causal attention among them and over the keys already cached.
//
// "qwen3-8b-rtx4080-cutedsl" README, "Flash Attention 2": the prompt's attention
// runs tile by tile with an online softmax, never forming the n x n score
// matrix; "Baseline tiled GEMM": the projections of the n rows are one GEMM per
// weight matrix (csrc/gemm_tc.cu, one CTA per 128 weight rows x 64 tokens).
//
// Attention layout on GB300: one CTA per (64 query rows, q head), four warps of
// 16 rows each. The queries (QK-RMSNorm, RoPE at their own positions, the
// softmax scale folded in) are staged once in shared memory as bf16 hi + lo
// parts, so q keeps ~16 mantissa bits through the bf16 MMAs; K/V tiles of 64
// keys stream through a two-stage cp.async ring into rows XOR-swizzled by 16-byte
// chunk (chunk c of row r at c ^ (r & 7)), which keeps every ldmatrix free of bank
// conflicts. Per tile and warp: S[16 x 64] = Q K^T (mma.sync m16n8k16, q hi and lo),
// the causal mask (key position <= the row's position), the online softmax in
// f32 (exp2 domain), and O[16 x 128] += P V with P taken straight from the S
// accumulators as the A operand (bf16 hi + lo) and V through transposing ldmatrix.
// Tiles past a warp's last row are skipped. The key range of a CTA ends at the
// position of its last row; K/V of the prompt itself are written to the cache by
// the K/V-write kernel before this one runs.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <cstdlib>

#include <algorithm>

namespace qd {
namespace {

constexpr int kPD = 128;               // head dimension
constexpr int kPQ = 64;                // query rows per CTA
constexpr int kPK = 64;                // keys per tile
constexpr int kPW = 4;                 // warps (16 query rows each)
constexpr int kPTh = kPW * 32;
constexpr int kPTile = kPK * kPD * 2;  // 16 KB per K or V tile
constexpr int kPStages = 2;
constexpr size_t kPSmem = 1024 + 2 * (size_t)kPQ * kPD * 2 + (size_t)kPStages * 2 * kPTile;

struct PfParams {
  const float* qkv;                    // f32 [n, (Hq + 2 Hkv) D]
  int n, Hq, Hkv;
  const __nv_bfloat16* q_norm;
  const float2* rope;
  int rope_max_pos;
  float eps;
  int act_bf16;
  const int32_t* pos;                  // pos[0]: the first prompt token's position
  const __nv_bfloat16* k_pages;
  const __nv_bfloat16* v_pages;
  const int32_t* page_table;           // the sequence's row
  int page_size, max_pages, n_pages;
  float scale_log2;
  __nv_bfloat16* out;                  // bf16 [n, Hq D]
  int* err;
};

QD_DEV void pf_mma(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
QD_DEV void pf_ldsm(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
QD_DEV void pf_ldsm_t(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
QD_DEV void pf_cp16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
QD_DEV void pf_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
QD_DEV void pf_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// byte offset of (row r, 16-byte chunk c) in a tile of 256-byte rows
QD_DEV uint32_t pf_swz(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4)); }

QD_DEV uint32_t pack_bf16(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// keys [t, t + kPK) of kv head g into one K and one V tile (keys at or past kend
// zero-filled)
QD_DEV void pf_load_tile(const PfParams& p, int g, int t, int kend, uint32_t sK, uint32_t sV) {
#pragma unroll
  for (int j = 0; j < (kPK * 16) / kPTh; ++j) {
    const int i = threadIdx.x + j * kPTh;
    const int r = i >> 4, c = i & 15;
    const int key = t + r;
    const bool ok = key < kend;
    size_t off = 0;
    if (ok) {
      const PagedSlot sl = paged_slot(p.page_table, key, p.page_size, p.n_pages);
      if (!sl.ok) set_error(p.err, QD_DEVERR_PAGE);
      else off = (((size_t)sl.page * p.Hkv + g) * p.page_size + sl.slot) * kPD + c * 8;
    }
    pf_cp16(sK + pf_swz(r, c), p.k_pages + off, ok ? 16 : 0);
    pf_cp16(sV + pf_swz(r, c), p.v_pages + off, ok ? 16 : 0);
  }
}

// PLO: P as bf16 hi + lo (two MMAs per P fragment) or its bf16 value alone.
template <bool PLO>
__global__ void __launch_bounds__(kPTh) prefill_attn_kernel(const PfParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sQh = smem;                          // [64 rows][256 B], swizzled
  unsigned char* sQl = sQh + kPQ * kPD * 2;
  unsigned char* ring = sQl + kPQ * kPD * 2;          // [stage][K, V]
  // the last query tiles see the most keys: launch them first so the short ones fill the tail
  const int qt = (int)(gridDim.x - 1 - blockIdx.x), h = blockIdx.y;
  const int g = h / (p.Hq / p.Hkv);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  pdl_wait();   // q, k, v of the prompt come from the kernels before this one
  pdl_launch_dependents();
  const int pos0 = p.pos[0];
  const int cap = p.max_pages * p.page_size;
  if (pos0 < 0 || pos0 + p.n > cap || pos0 + p.n > p.rope_max_pos) {
    if (qt == 0 && h == 0 && tid == 0) set_error(p.err, QD_DEVERR_POS);
    return;
  }
  const int r0 = qt * kPQ;
  const int nrows = min(kPQ, p.n - r0);
  const int kend = pos0 + r0 + nrows;                 // keys [0, kend) are visible to some row
  const int n_kt = (kend + kPK - 1) / kPK;
  const uint32_t ring_u = smem_u32(ring);
  auto tK = [&](int st) { return ring_u + (uint32_t)(st * 2 * kPTile); };
  auto tV = [&](int st) { return ring_u + (uint32_t)(st * 2 * kPTile + kPTile); };
  pf_load_tile(p, g, 0, kend, tK(0), tV(0));
  pf_commit();

  // ---- queries: warp w builds rows 16w .. 16w + 15; lane holds dims 4 lane .. + 3.
  // Four rows at a time: their activations and RoPE rows are all requested before
  // any is used, so a warp waits for four L2 round trips instead of 32.
  {
    const int qkv_w = (p.Hq + 2 * p.Hkv) * kPD;
    const int d0 = 4 * lane;
    const uint2 wq = *(const uint2*)(p.q_norm + d0);
    const float nw[4] = {bf_lo(wq.x), bf_hi(wq.x), bf_lo(wq.y), bf_hi(wq.y)};
    constexpr int kRB = 4;
    for (int rb = 0; rb < 16; rb += kRB) {
      float4 xr[kRB];
      float4 cr[kRB][2];
#pragma unroll
      for (int i = 0; i < kRB; ++i) {
        const int row = r0 + warp * 16 + rb + i;
        if (row < p.n) {
          xr[i] = *(const float4*)(p.qkv + (size_t)row * qkv_w + (size_t)h * kPD + d0);
          const float4* cs = (const float4*)(p.rope + (size_t)(pos0 + row) * (kPD / 2) + (d0 & 63));
          cr[i][0] = cs[0];
          cr[i][1] = cs[1];
        } else {
          xr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          cr[i][0] = cr[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int i = 0; i < kRB; ++i) {
        const int lr = warp * 16 + rb + i, row = r0 + lr;
        float qv[4] = {0.f, 0.f, 0.f, 0.f};
        if (row < p.n) {   // uniform over the warp
          const float xs[4] = {xr[i].x, xr[i].y, xr[i].z, xr[i].w};
          const float ss = warp_sum(xs[0] * xs[0] + xs[1] * xs[1] + xs[2] * xs[2] + xs[3] * xs[3]);
          const float inv = 1.0f / sqrtf(ss / (float)kPD + p.eps);
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
          lo[e] = pack_bf16(qv[2 * e] - __bfloat162float(h0), qv[2 * e + 1] - __bfloat162float(h1));
        }
        const uint32_t o = pf_swz(lr, lane >> 1) + (uint32_t)((lane & 1) * 8);
        *(uint2*)(sQh + o) = make_uint2(hi[0], hi[1]);
        *(uint2*)(sQl + o) = make_uint2(lo[0], lo[1]);
      }
    }
  }
  __syncthreads();

  const int gq = lane >> 2, tq = lane & 3;
  const int wrow0 = r0 + warp * 16;                                  // this warp's first row
  const int rowpos0 = pos0 + wrow0 + gq, rowpos1 = rowpos0 + 8;      // positions of rows g, g + 8
  const bool v0 = wrow0 + gq < p.n, v1 = wrow0 + gq + 8 < p.n;
  const int wlast = pos0 + min(wrow0 + 15, p.n - 1);                 // last key any row of the warp sees
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[j][e] = 0.f;
  const uint32_t qh_u = smem_u32(sQh), ql_u = smem_u32(sQl);
  const int mi = lane >> 3, mr = lane & 7;

  for (int kt = 0; kt < n_kt; ++kt) {
    const int st = kt & 1;
    if (kt + 1 < n_kt) pf_load_tile(p, g, (kt + 1) * kPK, kend, tK(st ^ 1), tV(st ^ 1));
    pf_commit();
    pf_wait<1>();
    __syncthreads();
    const int ks0 = kt * kPK;
    if (ks0 <= wlast && wrow0 < p.n) {
      // ---- S = Q K^T for 16 rows x 64 keys
      float s[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
      const uint32_t sK = tK(st), sV = tV(st);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t ah[4], al[4];
        const uint32_t qa = pf_swz(warp * 16 + (mi & 1) * 8 + mr, 2 * kk + (mi >> 1));
        pf_ldsm(ah, qh_u + qa);
        pf_ldsm(al, ql_u + qa);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t b[4];
          pf_ldsm(b, sK + pf_swz(16 * j + (mi >> 1) * 8 + mr, 2 * kk + (mi & 1)));
          pf_mma(s[2 * j], ah[0], ah[1], ah[2], ah[3], b[0], b[1]);
          pf_mma(s[2 * j], al[0], al[1], al[2], al[3], b[0], b[1]);
          pf_mma(s[2 * j + 1], ah[0], ah[1], ah[2], ah[3], b[2], b[3]);
          pf_mma(s[2 * j + 1], al[0], al[1], al[2], al[3], b[2], b[3]);
        }
      }
      // ---- causal mask and the online softmax (rows g and g + 8 of the warp)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = ks0 + 8 * j + 2 * tq + e;
          if (!v0 || key > rowpos0) s[j][e] = -INFINITY;
          if (!v1 || key > rowpos1) s[j][2 + e] = -INFINITY;
          mx0 = fmaxf(mx0, s[j][e]);
          mx1 = fmaxf(mx1, s[j][2 + e]);
        }
      }
#pragma unroll
      for (int o2 = 1; o2 <= 2; o2 <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
      const float al1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s[j][e] = s[j][e] == -INFINITY ? 0.f : exp2f(s[j][e] - mn0);
          s[j][2 + e] = s[j][2 + e] == -INFINITY ? 0.f : exp2f(s[j][2 + e] - mn1);
          ps0 += s[j][e];
          ps1 += s[j][2 + e];
        }
      }
      l0 = l0 * al0 + ps0;
      l1 = l1 * al1 + ps1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= al0;
        o[j][1] *= al0;
        o[j][2] *= al1;
        o[j][3] *= al1;
      }
      // ---- O += P V: P (bf16 hi + lo, or bf16) from the S accumulators, 16 keys per step
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float* pa = s[2 * kk];
        const float* pb = s[2 * kk + 1];
        uint32_t ph[4], pl[4];
        const float pv[4][2] = {{pa[0], pa[1]}, {pa[2], pa[3]}, {pb[0], pb[1]}, {pb[2], pb[3]}};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat16 h0 = __float2bfloat16_rn(pv[i][0]), h1 = __float2bfloat16_rn(pv[i][1]);
          ph[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
          if (PLO) pl[i] = pack_bf16(pv[i][0] - __bfloat162float(h0), pv[i][1] - __bfloat162float(h1));
        }
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          uint32_t b[4];
          pf_ldsm_t(b, sV + pf_swz(16 * kk + (mi & 1) * 8 + mr, 2 * dp + (mi >> 1)));
          pf_mma(o[2 * dp], ph[0], ph[1], ph[2], ph[3], b[0], b[1]);
          if (PLO) pf_mma(o[2 * dp], pl[0], pl[1], pl[2], pl[3], b[0], b[1]);
          pf_mma(o[2 * dp + 1], ph[0], ph[1], ph[2], ph[3], b[2], b[3]);
          if (PLO) pf_mma(o[2 * dp + 1], pl[0], pl[1], pl[2], pl[3], b[2], b[3]);
        }
      }
    }
    __syncthreads();  // the stage is refilled by the next iteration's copies
  }
  pf_wait<0>();

  // ---- O / l, rows g and g + 8 of the warp
#pragma unroll
  for (int o2 = 1; o2 <= 2; o2 <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
  }
  const size_t ow = (size_t)p.Hq * kPD;
  if (v0) {
    __nv_bfloat16* out = p.out + (size_t)(wrow0 + gq) * ow + (size_t)h * kPD + 2 * tq;
#pragma unroll
    for (int j = 0; j < 16; ++j) *(uint32_t*)(out + 8 * j) = pack_bf16(o[j][0] / l0, o[j][1] / l0);
  }
  if (v1) {
    __nv_bfloat16* out = p.out + (size_t)(wrow0 + gq + 8) * ow + (size_t)h * kPD + 2 * tq;
#pragma unroll
    for (int j = 0; j < 16; ++j) *(uint32_t*)(out + 8 * j) = pack_bf16(o[j][2] / l1, o[j][3] / l1);
  }
}

// positions of the prompt's rows: vpos[i] = pos[0] + i
__global__ void prefill_prep_kernel(const int32_t* pos, int n, int32_t* vpos) {
  pdl_wait();
  pdl_launch_dependents();
  const int p0 = pos[0];
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) vpos[i] = p0 + i;
}

// before the argmax advance (which adds one): pos[0] += n - 1
__global__ void prefill_finish_kernel(int32_t* pos, int n) {
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) pos[0] += n - 1;
}

}  // namespace

cudaError_t launch_prefill_attention(const PrefillAttnArgs& a, const Launch& L) {
  if (a.n < 1 || a.D != kPD || a.Hkv < 1 || a.Hq % a.Hkv) return cudaErrorInvalidValue;
  PfParams p = {};
  p.qkv = a.qkv; p.n = a.n; p.Hq = a.Hq; p.Hkv = a.Hkv;
  p.q_norm = (const __nv_bfloat16*)a.q_norm; p.rope = (const float2*)a.rope; p.rope_max_pos = a.rope_max_pos;
  p.eps = a.eps; p.act_bf16 = a.act_bf16; p.pos = a.pos;
  p.k_pages = (const __nv_bfloat16*)a.k_pages; p.v_pages = (const __nv_bfloat16*)a.v_pages;
  p.page_table = a.page_table; p.page_size = a.page_size; p.max_pages = a.max_pages; p.n_pages = a.n_pages;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.out = (__nv_bfloat16*)a.out; p.err = L.err;
  // QD_PREFILL_P_HILO (read per call): 1 keeps P as bf16 hi + lo, 0 its bf16 value alone
  const char* hl = getenv("QD_PREFILL_P_HILO");
  const bool plo = hl == nullptr || atoi(hl) != 0;
  auto k = plo ? prefill_attn_kernel<true> : prefill_attn_kernel<false>;
  static bool attr_set[2] = {false, false};
  if (!attr_set[plo]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmem);
    if (e != cudaSuccess) return e;
    attr_set[plo] = true;
  }
  return launch_ex(k, dim3(ceil_div(a.n, kPQ), a.Hq), dim3(kPTh), kPSmem, L, p);
}

cudaError_t launch_prefill_prep(const int32_t* pos, int n, int32_t* vpos, const Launch& L) {
  return launch_ex(prefill_prep_kernel, dim3(std::max(1, std::min(64, ceil_div(n, 256)))), dim3(256), 0, L, pos, n,
                   vpos);
}

cudaError_t launch_prefill_finish(int32_t* pos, int n, const Launch& L) {
  return launch_ex(prefill_finish_kernel, dim3(1), dim3(32), 0, L, pos, n);
}

}  // namespace qd
