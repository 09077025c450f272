// Small-batch weight-streaming GEMV on the tensor cores: y[b, r] = sum_k W[r, k] x[b, k]
// for B = 1..8 activation rows (the sequences of a small decode batch, or the k
// drafted tokens of one speculative-verify pass).
//
// "qwen3-8b-rtx4080-cutedsl" README, "Speculative decoding": verifying k drafted
// tokens runs every projection over k activation rows, and costs about one decode
// step's weight traffic when each weight is read once for all k rows. "GPU Kernel
// Lab" README, "Fundamental kernels": a decode GEMV is bound by the weight stream.
//
// GB300 layout of the work (the batch-1 ring GEMV's streaming, with the multiply-add
// on the tensor cores): one CTA per SM over a contiguous block of rows. A producer
// warp streams stages of 8 weight rows x PK columns through a shared-memory ring,
// issued before the programmatic-dependent wait because weights never depend on an
// earlier kernel. When a row fits in a stage the 8 rows are one contiguous copy;
// otherwise each row is its own 4 or 8 KB copy into rows an odd multiple of 64 bytes
// apart, so the consumers' 16-byte loads hit every bank once. (Copies of 1 KB held
// the stream near 3.2 TB/s on GB300, 2 KB near 5.4: the copy engine's per-copy cost
// sets the rate below about 4 KB.) Eight consumer warps split each stage's columns
// in 32-column chunks and run mma.sync m16n8k16 (bf16 in, f32 accumulate) with the
// activations as the 16-row A operand (rows 8..15 zero) and the 8 weight rows as the
// 8-column B operand: lane (g, t) loads columns 8t .. 8t + 7 of weight row g and of
// activation row g, the same pairing on both sides, so every product is a bf16 x
// bf16 product summed in binary32. A warp keeps the activation fragments of 4096
// columns in registers (16 per lane): K up to 4096 reads x once per CTA; a wider K
// runs range by range over all of a CTA's row groups (up to 64 rows, their sums in
// registers), so x is read once per CTA there too. The warps' partial sums reduce in
// a fixed order through shared memory, 32 rows at a time.
//
// Prologue: x as bf16 rows, or RMSNorm of f32 residual rows (bf16(w * bf16(x / rms))
// per element, the rounding of the row-normalisation kernel). Epilogue: store,
// residual add, or the SwiGLU pair form (W = [gate F rows; up F rows]; each CTA takes
// matching gate and up rows and writes h[b, j] = bf16(silu(g) * u)).
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <algorithm>
#include <cstdlib>

namespace qd {
namespace {

constexpr int kWarps = 8;                 // consumer warps
constexpr int kCons = 32 * kWarps;
constexpr int kSR = 8;                    // weight rows per stage (the MMA's N)
constexpr int kWin = 32;                  // rows reduced over the warps at a time
constexpr int kKR = 4096;                 // columns of activation fragments held in registers
constexpr int kXR = kKR / (32 * kWarps);  // fragments per lane (16)
constexpr int kMaxB = 8;
constexpr int kMaxStages = 16;
constexpr int kMaxRgQ = 8;                // row groups kept in registers across register ranges

struct MmaParams {
  const __nv_bfloat16* W;
  int R, K, B;
  int rows_base, rows_extra;   // CTA row partition (pairs under EPI_SWIGLU)
  int pair_F;                  // EPI_SWIGLU: rows of each half
  int pair_cap;                // EPI_SWIGLU: room per activation row for the CTA's sums
  int ns, stage_bytes, rstride, ring_bytes;
  int contig;                  // K fits a stage: a stage's rows are one contiguous copy
  int pro;
  const void* x;
  const __nv_bfloat16* norm_w;
  float eps;
  int epi;
  float* y;
  __nv_bfloat16* y_bf16;
  int* err;
  int w_evict_first;
  L2Prefetch pf;
};

QD_DEV void cons_sync_m() { asm volatile("bar.sync 1, %0;" ::"n"(kCons) : "memory"); }

// D += A B with A rows 8..15 zero (a1 = a3 = 0)
QD_DEV void mma_a8(float* d, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

QD_DEV uint32_t pack2(float lo, float hi) { return f2bf_bits(lo) | (f2bf_bits(hi) << 16); }

// Activation fragments of lane (g, t) of warp w for columns [k0, k0 + kKR): fragment j
// holds columns 8t .. 8t + 7 of 32-column chunk w + 8j, activation row g; zero past K
// or past the B rows.
QD_DEV void load_x(const MmaParams& p, int k0, int w, int g, int t, const float* s_inv, uint4 (&xr)[kXR]) {
#pragma unroll
  for (int j = 0; j < kXR; ++j) {
    const int col = k0 + 32 * (w + kWarps * j) + 8 * t;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (g < p.B && col < p.K) {
      if (p.pro == PRO_X_BF16) {
        v = *(const uint4*)((const __nv_bfloat16*)p.x + (size_t)g * p.K + col);
      } else {  // PRO_RMSNORM
        const float* xp = (const float*)p.x + (size_t)g * p.K + col;
        const float4 a = *(const float4*)xp, c = *(const float4*)(xp + 4);
        const uint4 nw = *(const uint4*)(p.norm_w + col);
        const float inv = s_inv[g];
        v.x = pack2(bf_lo(nw.x) * round_bf16(a.x * inv), bf_hi(nw.x) * round_bf16(a.y * inv));
        v.y = pack2(bf_lo(nw.y) * round_bf16(a.z * inv), bf_hi(nw.y) * round_bf16(a.w * inv));
        v.z = pack2(bf_lo(nw.z) * round_bf16(c.x * inv), bf_hi(nw.z) * round_bf16(c.y * inv));
        v.w = pack2(bf_lo(nw.w) * round_bf16(c.z * inv), bf_hi(nw.w) * round_bf16(c.w * inv));
      }
    }
    xr[j] = v;
  }
}

// CPW: 32-column chunks per warp per stage (a stage spans PK = 256 * CPW columns).
template <int CPW>
__global__ void __launch_bounds__(kCons + 32, 1) gemv_mma_kernel(const MmaParams p) {
  constexpr int PK = 32 * kWarps * CPW;
  constexpr int kPPR = kKR / PK;   // stages per register range
  static_assert(kKR % PK == 0, "a register range holds whole stages");
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = (uint64_t*)(smem + p.ring_bytes);
  uint64_t* empty = full + kMaxStages;
  float* red = (float*)(empty + kMaxStages);        // [kWarps][kWin rows][kMaxB]
  float* s_pair = red + kWarps * kWin * kMaxB;       // EPI_SWIGLU: [B][pair_cap]
  __shared__ float s_inv[kMaxB];
  __shared__ float s_ss[kWarps][kMaxB];
  __shared__ int s_fail;

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int K = p.K, ns = p.ns;
  const bool pair = p.epi == EPI_SWIGLU;
  const int nown = p.rows_base + ((int)blockIdx.x < p.rows_extra ? 1 : 0);
  const int npair = pair ? nown : 0;
  const int nrows = pair ? 2 * nown : nown;
  const int r0 = (int)blockIdx.x * p.rows_base + min((int)blockIdx.x, p.rows_extra);
  const int nrg = (nrows + kSR - 1) / kSR;
  const int npk = (K + PK - 1) / PK;                 // stages per row group
  const int n_stages = nrg * npk;
  // local row lr of the CTA -> weight row (the SwiGLU form's up rows follow the gate rows)
  auto wrow = [&](int lr) -> size_t {
    return (pair && lr >= npair) ? (size_t)p.pair_F + r0 + (lr - npair) : (size_t)r0 + lr;
  };

  if (tid == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kWarps);
    }
    s_fail = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  // Stage order. K up to 4096: row group by row group, each over its K range. Wider K
  // with at most kMaxRgQ row groups: register range by register range (4096 columns),
  // each over every row group, so the activation fragments load once per range and the
  // row groups' sums stay in registers; otherwise row group by row group with the
  // fragments reloaded per range.
  const int nq = (K + kKR - 1) / kKR;
  const bool qouter = nq > 1 && nrg <= kMaxRgQ;

  if (w == kWarps) {  // ---- producer warp: weights only, so no dependency wait
    const uint64_t pol = policy_evict_first();
    auto copy = [&](void* d, const void* s, uint32_t n, uint64_t* bar) {
      if (p.w_evict_first) bulk_g2s_hint(d, s, n, bar, pol);
      else bulk_g2s(d, s, n, bar);
    };
    int i = 0;
    auto issue = [&](int rg, int kp) -> bool {  // stage i: rows of group rg, columns of part kp
      const int slot = i % ns;
      int ok = 1;
      if (lane == 0 && i >= ns) ok = mbar_wait_bounded(&empty[slot], (uint32_t)(((i / ns) - 1) & 1), p.err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      const int a = rg * kSR;
      const int rows_i = min(kSR, nrows - a);
      const int k0 = kp * PK;
      const uint32_t bytes = (uint32_t)(min(PK, K - k0) * 2);
      unsigned char* dst = ring + (size_t)slot * p.stage_bytes;
      if (p.contig) {  // whole rows: one copy per run of consecutive weight rows
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[slot], (uint32_t)rows_i * bytes);
          const int na = pair ? max(0, min(a + rows_i, npair) - a) : rows_i;   // rows before the up half
          if (na > 0) copy(dst, p.W + wrow(a) * K, (uint32_t)na * bytes, &full[slot]);
          if (rows_i > na) copy(dst + (size_t)na * bytes, p.W + wrow(a + na) * K, (uint32_t)(rows_i - na) * bytes,
                                &full[slot]);
        }
      } else {
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)rows_i * bytes);
        __syncwarp();
        if (lane < rows_i) copy(dst + (size_t)lane * p.rstride, p.W + wrow(a + lane) * K + k0, bytes, &full[slot]);
      }
      ++i;
      return true;
    };
    if (qouter) {
      bool go = true;
      for (int q = 0; q < nq && go; ++q)
        for (int rg = 0; rg < nrg && go; ++rg)
          for (int pp = 0; pp < kPPR && go; ++pp) {
            const int kp = q * kPPR + pp;
            if (kp * PK >= K) break;
            go = issue(rg, kp);
          }
    } else {
      bool go = true;
      for (int rg = 0; rg < nrg && go; ++rg)
        for (int kp = 0; kp < npk && go; ++kp) go = issue(rg, kp);
    }
    // the ring's last refills are in flight: DRAM would idle while the consumers
    // drain, so fetch the head of the next GEMV's spans into L2
    l2_prefetch_spans(p.pf, blockIdx.x, gridDim.x, lane);
    return;
  }

  // ---- consumers
  const int g = lane >> 2, t = lane & 3;
  pdl_wait();
  if (p.pro == PRO_RMSNORM) {
    // 1 / rms of every activation row. Lane (g, t) of warp w reads exactly the columns
    // of row g its fragments hold (every column of every row once over the CTA), all
    // loads in flight; sums over the four lanes of a row, then over the warps. load_x
    // reads the same addresses again (L1 hits).
    float ss = 0.f;
    for (int q = 0; q < nq; ++q) {
      float4 v[kXR][2];
#pragma unroll
      for (int j = 0; j < kXR; ++j) {
        const int col = q * kKR + 32 * (w + kWarps * j) + 8 * t;
        const bool in = g < p.B && col < K;
        const float* xp = (const float*)p.x + (size_t)g * K + col;
        v[j][0] = in ? *(const float4*)xp : make_float4(0.f, 0.f, 0.f, 0.f);
        v[j][1] = in ? *(const float4*)(xp + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kXR; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          ss = fmaf(v[j][h].x, v[j][h].x, ss);
          ss = fmaf(v[j][h].y, v[j][h].y, ss);
          ss = fmaf(v[j][h].z, v[j][h].z, ss);
          ss = fmaf(v[j][h].w, v[j][h].w, ss);
        }
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    if (t == 0) s_ss[w][g] = ss;
    cons_sync_m();
    if (tid < p.B) {
      float tot = 0.f;
#pragma unroll
      for (int k = 0; k < kWarps; ++k) tot += s_ss[k][tid];
      s_inv[tid] = 1.0f / sqrtf(tot / (float)K + p.eps);
    }
    cons_sync_m();
  }

  const size_t cstride = p.contig ? (size_t)K * 2 : (size_t)p.rstride;   // bytes between a stage's rows
  uint4 xr[kXR];
  int i = 0;          // stage counter
  bool ok = true;
  // One stage: MMAs of this warp's chunks of stage i (columns k0 ..) into acc, with the
  // activation fragments xbase .. of the current range. false: the wait gave up.
  auto run_stage = [&](int k0, int xbase, float* acc) -> bool {
    const int slot = i % ns;
    if (!mbar_wait_bounded(&full[slot], (uint32_t)((i / ns) & 1), p.err)) {
      // drain the copies that may still land in this CTA's ring, then stop
      for (int k = 1; k < ns && i + k < n_stages; ++k)
        mbar_wait_limit(&full[(i + k) % ns], (uint32_t)(((i + k) / ns) & 1), p.err, 10000000ull);
      return false;
    }
    const unsigned char* wp = ring + (size_t)slot * p.stage_bytes + (size_t)g * cstride + t * 16;
#pragma unroll
    for (int ci = 0; ci < CPW; ++ci) {
      const int cl = w + kWarps * ci;            // chunk of the stage
      if (k0 + 32 * cl >= K) break;              // the same for the whole warp
      const uint4 xf = xr[xbase + ci];
      const uint4 wv = *(const uint4*)(wp + cl * 64);
      mma_a8(acc, xf.x, xf.y, wv.x, wv.y);
      mma_a8(acc, xf.z, xf.w, wv.z, wv.w);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    ++i;
    return true;
  };
  // Row group rg's sums (activation row g; weight rows 2t, 2t + 1 of the group) into the
  // window; when the window is full or rg is the last group, the fixed-order sum over
  // the warps and the epilogue. false: a wait gave up in some warp (all return).
  auto put = [&](int rg, float a0, float a1) -> bool {
    const int wr = (rg % (kWin / kSR)) * kSR;       // first row of this group in the window
    float* rw = red + w * (kWin * kMaxB);
    rw[(wr + 2 * t) * kMaxB + g] = a0;
    rw[(wr + 2 * t + 1) * kMaxB + g] = a1;
    if (wr + kSR < kWin && rg + 1 < nrg) return true;   // the window is not full yet
    if (!ok && lane == 0) s_fail = 1;
    cons_sync_m();
    if (s_fail) return false;   // every consumer warp sees the same flag after the barrier
    const int wbase = rg * kSR - wr;                 // first local row of the window
    const int rows = min(kWin, nrows - wbase);
    for (int idx = tid; idx < p.B * kWin; idx += kCons) {
      const int b = idx / kWin, lr = idx - b * kWin;
      if (lr >= rows) continue;
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < kWarps; ++k) s += red[(k * kWin + lr) * kMaxB + b];
      const int row = wbase + lr;
      if (pair) {
        s_pair[b * p.pair_cap + row] = s;
      } else {
        float* yp = p.y + (size_t)b * p.R + r0 + row;
        if (p.epi == EPI_RESID_ADD) *yp += s;
        else *yp = s;
      }
    }
    cons_sync_m();
    return true;
  };

  if (qouter) {
    // C fragment per row group: [0] = (activation row g, weight row 2t), [1] = (g, 2t + 1)
    float acc[kMaxRgQ][4];
#pragma unroll
    for (int r = 0; r < kMaxRgQ; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[r][e] = 0.f;
    for (int q = 0; q < nq && ok; ++q) {
      load_x(p, q * kKR, w, g, t, s_inv, xr);
#pragma unroll
      for (int rg = 0; rg < kMaxRgQ; ++rg) {
        if (rg >= nrg || !ok) break;
#pragma unroll
        for (int pp = 0; pp < kPPR; ++pp) {
          const int k0 = q * kKR + pp * PK;
          if (k0 >= K) break;
          if (!run_stage(k0, pp * CPW, acc[rg])) {
            ok = false;
            break;
          }
        }
      }
    }
#pragma unroll
    for (int rg = 0; rg < kMaxRgQ; ++rg) {
      if (rg >= nrg) break;
      if (!put(rg, acc[rg][0], acc[rg][1])) return;
    }
  } else {
    for (int rg = 0; rg < nrg; ++rg) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int q = 0; q < nq && ok; ++q) {
        if (nq > 1 || rg == 0) load_x(p, q * kKR, w, g, t, s_inv, xr);
#pragma unroll
        for (int pp = 0; pp < kPPR; ++pp) {
          const int k0 = q * kKR + pp * PK;
          if (k0 >= K) break;
          if (!run_stage(k0, pp * CPW, acc)) {
            ok = false;
            break;
          }
        }
      }
      if (!put(rg, acc[0], acc[1])) return;
    }
  }
  if (pair) {  // SwiGLU of the CTA's pairs (the last window ended with a barrier)
    for (int idx = tid; idx < p.B * npair; idx += kCons) {
      const int b = idx / npair, j = idx - b * npair;
      const float gg = s_pair[b * p.pair_cap + j], uu = s_pair[b * p.pair_cap + npair + j];
      p.y_bf16[(size_t)b * p.pair_F + r0 + j] = __float2bfloat16_rn(gg / (1.0f + expf(-gg)) * uu);
    }
  }
}

struct MmaTuning {
  int cpw;       // QD_MMA_CPW: 8 (2048-column stages) or 16 (4096)
  int ring_kb;   // QD_MMA_RING_KB: ring bytes target
};
const MmaTuning& mma_tuning() {
  static const MmaTuning t = [] {
    MmaTuning r;
    const char* v = getenv("QD_MMA_CPW");
    r.cpw = (v && atoi(v) == 8) ? 8 : 16;
    v = getenv("QD_MMA_RING_KB");
    r.ring_kb = v ? std::max(32, atoi(v)) : 200;
    return r;
  }();
  return t;
}

template <int CPW>
cudaError_t launch_mma_c(const MmaParams& p, int grid, size_t smem, const Launch& L) {
  auto k = gemv_mma_kernel<CPW>;
  static bool attr_set = false;
  if (!attr_set) {
    // the launcher asks for at most this much (static shared memory comes on top)
    cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dev_info().max_smem_optin - 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(k, dim3(grid), dim3(kCons + 32), smem, L, p);
}

}  // namespace

bool gemv_mma_supported(int R, int K, int B) {
  return R >= 1 && B >= 1 && B <= kMaxB && K >= 32 && K % 32 == 0;
}

cudaError_t launch_gemv_mma(const GemvMmaArgs& a, const Launch& L) {
  const bool pair = a.epi == EPI_SWIGLU;
  if (!gemv_mma_supported(a.R, a.K, a.B) || (pair && (a.R % 2 != 0 || !a.y_bf16)) || (!pair && !a.y) ||
      (a.pro != PRO_X_BF16 && a.pro != PRO_RMSNORM) || (a.pro == PRO_RMSNORM && !a.norm_w))
    return cudaErrorInvalidValue;
  const MmaTuning& tu = mma_tuning();
  const int units = pair ? a.R / 2 : a.R;
  const int grid = std::min(dev_info().sm_count, units);
  MmaParams p = {};
  p.W = (const __nv_bfloat16*)a.W;
  p.R = a.R; p.K = a.K; p.B = a.B;
  p.rows_base = units / grid;
  p.rows_extra = units % grid;
  p.pair_F = pair ? a.R / 2 : 0;
  p.pair_cap = pair ? 2 * (p.rows_base + 1) : 0;
  const int pk = 256 * tu.cpw;
  p.contig = a.K <= pk;
  if (p.contig) {
    p.rstride = a.K * 2;
  } else {  // an odd multiple of 64 bytes between the rows of a stage
    p.rstride = ((pk * 2 + 127) / 128) * 128 + 64;
  }
  p.stage_bytes = ((kSR * p.rstride + 127) / 128) * 128;
  const size_t fixed = (size_t)2 * kMaxStages * 8 + (size_t)kWarps * kWin * kMaxB * 4 +
                       (size_t)kMaxB * p.pair_cap * 4;
  const size_t avail = (size_t)dev_info().max_smem_optin - 1024 - fixed;
  const size_t want = std::min(avail, (size_t)tu.ring_kb * 1024);
  p.ns = (int)std::min<size_t>(kMaxStages, want / p.stage_bytes);
  if (p.ns < 2) return cudaErrorInvalidValue;
  p.ring_bytes = p.ns * p.stage_bytes;
  p.pro = a.pro; p.x = a.x; p.norm_w = (const __nv_bfloat16*)a.norm_w; p.eps = a.eps;
  p.epi = a.epi; p.y = a.y; p.y_bf16 = (__nv_bfloat16*)a.y_bf16;
  p.err = L.err;
  p.w_evict_first = a.w_evict_first;
  p.pf = a.pf;
  const size_t smem = (size_t)p.ring_bytes + fixed;
  return tu.cpw == 8 ? launch_mma_c<8>(p, grid, smem, L) : launch_mma_c<16>(p, grid, smem, L);
}

}  // namespace qd
