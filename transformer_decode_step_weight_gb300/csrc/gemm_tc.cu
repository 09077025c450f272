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
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

namespace qd {
namespace {

constexpr int kBM = 128;        // weight rows per tile (MMA M)
constexpr int kBN = 64;         // tokens (MMA N, TMEM columns)
constexpr int kBK = 64;         // K elements per stage (128 bytes of bf16)
// Ring depth: 6 stages (one CTA per SM) when the CTAs fit in one wave, else 3
// (~74 KB, two or three CTAs per SM, so a grid of up to twice the SM count still
// runs in one wave). QD_GEMM_STAGES = 3 or 6 forces one.
constexpr int kTileA = kBM * kBK * 2;    // 16 KB
constexpr int kTileB = kBN * kBK * 2;    // 8 KB
constexpr int kThreadsTc = 128;
constexpr int kMaxSplits = 4;   // K splits of one tile (partials summed in registers)

struct TcParams {
  int R, K, B;
  int epi;        // EPI_STORE / EPI_RESID_ADD
  float* y;       // [B, R]
  int* err;
  int splits;     // K splits (grid y); > 1: partials through part / cnt
  float* part;    // [tiles][splits][kBN][kBM] f32 partial tiles
  int* cnt;       // [tiles] tickets, zero between launches
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

// Instruction descriptor: D f32, A and B bf16, both K-major, M = 128, N = 64.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

QD_DEV void mma_bf16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t accumulate) {
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

template <int kStagesTc>
__global__ void __launch_bounds__(kThreadsTc, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sA = smem;                                   // [stages][128 x 128 B]
  unsigned char* sB = smem + kStagesTc * kTileA;              // [stages][64 x 128 B]
  uint64_t* full = (uint64_t*)(sB + kStagesTc * kTileB);
  uint64_t* empty = full + kStagesTc;
  uint64_t* done = empty + kStagesTc;
  uint32_t* tmem_slot = (uint32_t*)(done + 1);
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = blockIdx.x * kBM;
  // this CTA's K blocks [kb0, kb0 + n_k) of split blockIdx.y
  const int n_kt = p.K / kBK;
  const int kb0 = (int)(((long long)n_kt * blockIdx.y) / p.splits);
  const int n_k = (int)(((long long)n_kt * (blockIdx.y + 1)) / p.splits) - kb0;
  __shared__ int s_ticket;

  if (tid == 0) {
    for (int i = 0; i < kStagesTc; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(tmem_slot, kBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0 && lane == 0) {
    // ---- producer: W tiles need no dependency; X (this step's activations) does
    const int pre = min(kStagesTc, n_k);
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&full[i], kTileA + kTileB);
      tma_load_2d(sA + i * kTileA, &tmW, (kb0 + i) * kBK, row0, &full[i]);
    }
    pdl_wait();
    for (int i = 0; i < pre; ++i) tma_load_2d(sB + i * kTileB, &tmX, (kb0 + i) * kBK, 0, &full[i]);
    for (int i = pre; i < n_k; ++i) {
      const int s = i % kStagesTc;
      if (!mbar_wait_bounded(&empty[s], (uint32_t)(((i / kStagesTc) - 1) & 1), p.err)) {
        s_abort = 1;
        break;
      }
      mbar_arrive_expect_tx(&full[s], kTileA + kTileB);
      tma_load_2d(sA + s * kTileA, &tmW, (kb0 + i) * kBK, row0, &full[s]);
      tma_load_2d(sB + s * kTileB, &tmX, (kb0 + i) * kBK, 0, &full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    for (int i = 0; i < n_k; ++i) {
      const int s = i % kStagesTc;
      if (!mbar_wait_bounded(&full[s], (uint32_t)((i / kStagesTc) & 1), p.err)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA + s * kTileA), b0 = smem_u32(sB + s * kTileB);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        mma_bf16(tmem, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), (i | kk) != 0);
      mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
    }
    mma_commit(done);         // D complete (also arrives after an early exit)
  }
  __syncwarp();

  // ---- epilogue: warp w owns TMEM lanes [32w, 32w + 32) = rows row0 + 32w + lane
  pdl_wait();
  const bool ok = mbar_wait_bounded(done, 0, p.err);
  tc_fence_after();
  float v[64];
  tmem_ld_32x64(tmem + ((uint32_t)(warp * 32) << 16), v);
  const int rl = warp * 32 + lane;          // this thread's row of the tile
  const int r = row0 + rl;
  bool write = ok && !s_abort;
  // y[n0 + j, r] (+)= o[j] for 16 tokens; the residual values are all loaded
  // before any store, so the 16 read-modify-writes overlap instead of queueing
  auto store_rows = [&](int n0, const float* o) {
    float old[16];
    if (p.epi == EPI_RESID_ADD) {
#pragma unroll
      for (int j = 0; j < 16; ++j) old[j] = n0 + j < p.B ? p.y[(size_t)(n0 + j) * p.R + r] : 0.f;
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) old[j] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (n0 + j < p.B) p.y[(size_t)(n0 + j) * p.R + r] = p.epi == EPI_RESID_ADD ? old[j] + o[j] : o[j];
  };
  if (p.splits > 1) {
    // publish this split's partial tile [kBN tokens][kBM rows] (each warp access
    // one 128-byte line), take a ticket; the last split of the tile adds every
    // partial in split order, 16 tokens at a time with all their loads (and the
    // residual's) in flight together
    const size_t tile = blockIdx.x;
    float* part = p.part + (tile * p.splits + blockIdx.y) * (size_t)(kBN * kBM);
#pragma unroll
    for (int n = 0; n < kBN; ++n) part[(size_t)n * kBM + rl] = v[n];
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
  if (write && r < p.R) {
#pragma unroll
    for (int c = 0; c < kBN / 16; ++c) store_rows(c * 16, v + c * 16);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kBN);
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

// Row-major bf16 [rows, cols] matrix, box of box_rows x 64 columns, 128-byte swizzle.
cudaError_t encode_rowmajor_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                                 uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

constexpr size_t smem_tc(int st) { return 1024 + (size_t)st * (kTileA + kTileB) + (2 * st + 1) * 8 + 16; }

template <int ST>
cudaError_t launch_tc(const CUtensorMap& tw, const CUtensorMap& tx, const TcParams& p, int tiles, const Launch& L) {
  auto k = gemm_tc_kernel<ST>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_tc(ST));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_ex(k, dim3(tiles, p.splits), dim3(kThreadsTc), smem_tc(ST), L, tw, tx, p);
}

}  // namespace

cudaError_t encode_tmap_bf16_2d(void* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return encode_rowmajor_bf16((CUtensorMap*)map, base, rows, cols, box_rows);
}

bool gemm_tc_supported(int R, int K, int B) { return R >= 1 && K >= kBK && K % kBK == 0 && B >= 1 && B <= kBN; }

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

int gemm_tc_splits(int R, int K) {
  if (R < 1 || K < kBK) return 1;
  const int tiles = (R + kBM - 1) / kBM, n_kt = K / kBK, sms = dev_info().sm_count;
  if (tiles > kMaxSplitTiles) return 1;
  static const int forced = [] {
    const char* v = getenv("QD_GEMM_SPLITS");
    return v ? atoi(v) : 0;
  }();
  if (forced > 0) return std::max(1, std::min(std::min(forced, kMaxSplits), n_kt));
  if (tiles >= sms) return 1;  // the tiles alone fill the GPU (measured: splitting them was slower)
  int best = 1;
  double best_t = (double)((tiles + sms - 1) / sms);
  const double tile_bytes = (double)kBM * K * 2;
  for (int sp = 2; sp <= kMaxSplits && n_kt / sp >= 8; ++sp) {
    const double t = (double)((tiles * sp + sms - 1) / sms) / sp + 0.5 * sp * 65536.0 / tile_bytes;
    if (t < best_t) {
      best_t = t;
      best = sp;
    }
  }
  return best;
}

size_t gemm_tc_workspace_bytes(int R, int K) {
  const int sp = gemm_tc_splits(R, K);
  if (sp <= 1) return 0;
  const size_t tiles = (size_t)(R + kBM - 1) / kBM;
  return kTicketBytes + tiles * sp * kBN * kBM * sizeof(float);
}

cudaError_t launch_gemm_tc(const GemmTcArgs& a, const Launch& L) {
  if (!gemm_tc_supported(a.R, a.K, a.B)) return cudaErrorInvalidValue;
  CUtensorMap tw, tx;
  cudaError_t e = encode_rowmajor_bf16(&tw, a.W, (uint64_t)a.R, (uint64_t)a.K, kBM);
  if (e != cudaSuccess) return e;
  // X has B rows; the 64-row box reads zeros past them
  e = encode_rowmajor_bf16(&tx, a.X, (uint64_t)a.B, (uint64_t)a.K, kBN);
  if (e != cudaSuccess) return e;
  TcParams p = {};
  p.R = a.R; p.K = a.K; p.B = a.B; p.epi = a.epi; p.y = a.y; p.err = L.err;
  const int tiles = (a.R + kBM - 1) / kBM;
  p.splits = 1;
  const size_t need = gemm_tc_workspace_bytes(a.R, a.K);
  if (a.ws && need > 0 && a.ws_bytes >= need) {
    p.splits = gemm_tc_splits(a.R, a.K);
    p.cnt = (int*)a.ws;
    p.part = (float*)((unsigned char*)a.ws + kTicketBytes);
  }
  static const int forced = [] {
    const char* v = getenv("QD_GEMM_STAGES");
    return v ? atoi(v) : 0;
  }();
  const bool deep = forced == 6 || (forced != 3 && (long long)tiles * p.splits <= dev_info().sm_count);
  return deep ? launch_tc<6>(tw, tx, p, tiles, L) : launch_tc<3>(tw, tx, p, tiles, L);
}

}  // namespace qd
