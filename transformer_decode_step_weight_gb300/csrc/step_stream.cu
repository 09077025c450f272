// The whole decode step of a BF16 model at batch 1 as one persistent kernel.
//
// "GPU Kernel Lab" README, "Decode integration": the order of one step
// (projections, Q/K RMSNorm + RoPE + direct K/V cache write, split-KV GQA
// attention, residual + RMSNorm, gate/up + SwiGLU, down + residual, final
// RMSNorm + LM head + argmax with the token and position advanced on the
// device). "emit_qwen38_generate" rustdoc, "Where the speed comes from": one
// GEMV per shared activation, residual + RMSNorm fused into the next
// projection, one graph per token. "qwen3-8b-rtx4080-cutedsl" README,
// "Split-KV decode attention" and "GQA + QK-Norm".
//
// At batch 1 the step is a stream of weight bytes (15.1 GB for Qwen3-8B) with
// short dependent work between the projections. One kernel per projection
// leaves HBM idle at every kernel boundary and through the attention's latency
// chain. Here one CTA per SM runs the whole step:
//   * a producer warp walks this CTA's share of the step's byte stream in
//     order -- per layer its rows of W_qkv, its split of the K/V cache, its
//     rows of W_o, its gate/up row pairs of W_gu, its rows of W_down, then its
//     rows of the LM head -- through a 4-stage ring of 48 KB shared-memory
//     stages (weights by TMA bulk copy with an evict-first L2 policy; K/V as
//     16-token TMA tensor boxes in the 128-byte swizzle), and fetches the same
//     stream kPfAhead stages ahead into L2. It never waits for activations, so
//     HBM keeps streaming while the consumers wait on a dependency;
//   * eight consumer warps compute each phase from the ring: the projections as
//     warp-reduced GEMVs with this thread's activation slice in registers
//     (RMSNorm in the prologue, residual add or SwiGLU in the epilogue), the
//     attention split on the tensor cores (mma.sync, bf16 hi + lo parts of q
//     and P, f32 accumulation), the split combine by the last split of each kv
//     head (ticket), and the LM head with a running argmax;
//   * a phase that needs the whole output of an earlier one waits on a counter
//     in global memory that every contributing CTA increments, with release
//     ordering, once its part is written. One thread polls it with acquire
//     loads; the wait gives up after about a second (QD_DEVERR_TIMEOUT) and then
//     raises an abort word that ends every other CTA's waits at once;
//   * the grid is one CTA per SM, launched cooperatively, so every CTA is
//     resident and a wait never depends on a CTA that cannot be scheduled. The
//     last CTA through the argmax resets the counters for the next launch.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

#include <algorithm>
#include <climits>
#include <cstring>
#include <mutex>

namespace qd {
namespace {

constexpr int kCW = 8;                  // consumer warps
constexpr int kCT = kCW * 32;           // consumer threads
constexpr int kST = kCT + 32;           // plus the producer warp
#ifndef QD_STREAM_STAGE_KB
#define QD_STREAM_STAGE_KB 48
#endif
#ifndef QD_STREAM_STAGES
#define QD_STREAM_STAGES 4
#endif
#ifndef QD_STREAM_PF_AHEAD
#define QD_STREAM_PF_AHEAD 0
#endif
#ifndef QD_STREAM_PF_STALL
#define QD_STREAM_PF_STALL 0
#endif
constexpr int kStageB = QD_STREAM_STAGE_KB * 1024;  // bytes per ring stage
constexpr int kNSt = QD_STREAM_STAGES;              // ring stages
constexpr int kD = 128;                 // head dim
constexpr int kTokS = kStageB / (kD * 2 * 2);  // K/V tokens per stage (96)
constexpr int kFlush = 128;             // rows per reduction window
constexpr int kMaxSplit = 64;           // attention splits per kv head
constexpr int kMaxPair = 256;           // gate/up pairs per CTA
constexpr int kMaxOwnRows = 256;        // residual rows per CTA (kept in shared memory)
constexpr int kPfAhead = QD_STREAM_PF_AHEAD;  // stages the L2 read-ahead leads the copies by
constexpr int kPfStall = QD_STREAM_PF_STALL;  // ... and how far it may run on while stalled
constexpr int kHP = 8;                  // q heads padded to the MMA N
constexpr float kLog2e = 1.4426950408889634f;

// Profiling build only (-DQD_STREAM_TRACE): per-CTA global-timer stamps of every
// phase boundary, and of the producer's first copy of every item, into a buffer
// set by qd_stream_trace_set. The product build compiles none of this.
#ifdef QD_STREAM_TRACE
__device__ unsigned long long* g_stream_trace = nullptr;
constexpr int kTraceStride = 4096;  // events per CTA
#define STRACE(ev)                                                                      \
  do {                                                                                \
    if (g_stream_trace) g_stream_trace[(size_t)blockIdx.x * kTraceStride + (ev)] = global_ns(); \
  } while (0)
#else
#define STRACE(ev) \
  do {             \
  } while (0)
#endif

enum { IT_QKV = 0, IT_KV = 1, IT_O = 2, IT_GU = 3, IT_DOWN = 4, IT_LM = 5, IT_END = 6 };
enum { PH_QKV = 0, PH_ATTN = 1, PH_O = 2, PH_GU = 3, PH_DOWN = 4 };

struct SLayer {
  const __nv_bfloat16 *w_qkv, *w_o, *w_gu, *w_down, *ln_in, *ln_post, *q_norm, *k_norm;
  __nv_bfloat16 *k_cache, *v_cache;
};

struct SParams {
  SLayer L[kStreamMaxLayers];
  int n_layers, H, Hq, Hkv, F, V, rep;
  float eps, scale_log2;
  const __nv_bfloat16 *embed, *final_norm, *lm_head;
  const int32_t* page_table;
  int page_size, max_pages, n_pages;
  const float2* rope;
  int rope_max_pos;
  int32_t *tok, *pos, *step, *out_tokens;
  int max_steps;
  float* logits;
  float* res;                 // f32 [H]
  float* qkv;                 // f32 [(Hq + 2 Hkv) D]
  __nv_bfloat16* attn;        // bf16 [Hq D]
  __nv_bfloat16* h;           // bf16 [F]
  float* part;                // [Hkv][kMaxSplit][rep][D] split partials
  float* part_ml;             // [Hkv][kMaxSplit][rep][2] (max, sum)
  int* sync;                  // [5 L] phase counters, [64] tickets, argmax ticket, abort word
  float* cand_v;              // [grid] argmax candidates
  int* cand_i;
  int* err;
};

struct STmaps {
  CUtensorMap k[kStreamMaxLayers];
  CUtensorMap v[kStreamMaxLayers];
};

// ---------------------------------------------------------------- shared memory
struct Carve {
  static constexpr size_t ring = 0;
  static constexpr size_t bars = ring + (size_t)kNSt * kStageB;        // full[kNSt], empty[kNSt]
  static constexpr size_t red = bars + 2 * kNSt * 8;                   // [kFlush][8] f32; combine scratch
  static constexpr size_t pair = red + (size_t)kFlush * 8 * 4;         // [2 kMaxPair] f32
  static constexpr size_t misc = pair + (size_t)2 * kMaxPair * 4;      // 16 f32 + 16 int
  static constexpr size_t qh = misc + 128;                             // [8][128] bf16
  static constexpr size_t ql = qh + kHP * kD * 2;
  static constexpr size_t pbuf = ql + kHP * kD * 2;                    // [kCW][2][8][16] bf16
  static constexpr size_t ml = pbuf + (size_t)kCW * 2 * kHP * 16 * 2;  // [2][kCW][8] f32
  static constexpr size_t ared = ml + 2 * kCW * kHP * 4;               // [4][9] f32 + [128] f32
  static constexpr size_t obuf = ared + 64 * 4 + kD * 4;               // [kCW][4][128] f32 (q staging first)
  static constexpr size_t resown = obuf + (size_t)kCW * 4 * kD * 4;  // [kMaxOwnRows] f32
  static constexpr size_t total = resown + (size_t)kMaxOwnRows * 4;
};
constexpr size_t kSmemBytes = Carve::total + 1024;  // + alignment slack of the ring

struct Smem {
  unsigned char* ring;
  uint64_t* full;
  uint64_t* empty;
  float* red;
  float* pair;
  float* misc_f;
  int* misc_i;
  __nv_bfloat16* qh;
  __nv_bfloat16* ql;
  __nv_bfloat16* pb;
  float* sM;
  float* sL;
  float* ared;
  float* sx;
  float* obuf;
  float* resown;  // this CTA's rows of the residual (the rows its O and down phases own)
};

// ---------------------------------------------------------------- sync primitives
QD_DEV void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory"); }
// consumer barrier that also ANDs a predicate over the consumer threads
QD_DEV bool cbar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kCT)
      : "memory");
  return r != 0;
}
QD_DEV void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
QD_DEV int atom_acq_rel_add(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
QD_DEV int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// one thread: wait until *cnt >= target; false after about a second (error bit and
// the abort word set) or at once when another CTA has raised the abort word
QD_DEV bool wait_count(const int* cnt, int target, int* abort_w, int* err) {
  if (ld_acquire(cnt) >= target) return true;
  const uint64_t t0 = global_ns();
  for (int i = 0; i < (1 << 24); ++i) {
    if (ld_acquire(cnt) >= target) return true;
    if ((i & 31) == 31) {
      if (ld_acquire(abort_w) != 0) return false;
      if (global_ns() - t0 > 1000000000ull) break;
    }
    __nanosleep(64);
  }
  set_error(err, QD_DEVERR_TIMEOUT);
  atomicExch(abort_w, 1);
  return false;
}

// ---------------------------------------------------------------- the stream schedule
struct Span {
  int r0, n;
};
// the share of R units of CTA c: contiguous, sizes differing by at most one
QD_DEV Span span_of(int R, int c, int n_cta) {
  const int grid = min(R, n_cta);
  if (c >= grid) return Span{0, 0};
  const int base = R / grid, extra = R % grid;
  return Span{c * base + min(c, extra), base + (c < extra ? 1 : 0)};
}

struct KvSplit {
  int g, s, n_split, t0, t1;  // g < 0: this CTA has no split
};
// Splits of 16-token granules: min(kMaxSplit, grid / Hkv) per kv head, at most one
// per granule, so every split holds at least one key.
QD_DEV KvSplit kv_split(int c, int n_cta, int Hkv, int len) {
  KvSplit k;
  const int n_gran = (len + 15) / 16;
  k.n_split = max(1, min(min(kMaxSplit, n_cta / Hkv), n_gran));
  if (c >= Hkv * k.n_split) {
    k.g = -1; k.s = 0; k.t0 = k.t1 = 0;
    return k;
  }
  k.g = c / k.n_split;
  k.s = c % k.n_split;
  const int a = (int)((long long)n_gran * k.s / k.n_split);
  const int b = (int)((long long)n_gran * (k.s + 1) / k.n_split);
  k.t0 = 16 * a;
  k.t1 = min(16 * b, len);
  return k;
}

struct Item {
  int kind, layer;
  // rows items (projections): span 1 then span 2 (gate+up: the up rows)
  const unsigned char* src1;
  const unsigned char* src2;
  int r0, n1, n2, row_bytes, rps, n_stages;
  // K/V item
  int g, s, n_split, t0, t1;
};

struct Ctx {
  int c, n_cta, pos, len;
};

QD_DEV void rows_item(Item& it, const __nv_bfloat16* W, int R, int K, const Ctx& x) {
  const Span sp = span_of(R, x.c, x.n_cta);
  it.row_bytes = K * 2;
  it.rps = min(kFlush, kStageB / it.row_bytes);
  it.r0 = sp.r0;
  it.n1 = sp.n;
  it.n2 = 0;
  it.src1 = (const unsigned char*)(W + (size_t)sp.r0 * K);
  it.src2 = nullptr;
  it.n_stages = (sp.n + it.rps - 1) / it.rps;
}

QD_DEV Item get_item(const SParams& p, const Ctx& x, int idx) {
  Item it = {};
  const int Lq = 5 * p.n_layers;
  if (idx > Lq) {
    it.kind = IT_END;
    return it;
  }
  if (idx == Lq) {
    it.kind = IT_LM;
    it.layer = p.n_layers;
    rows_item(it, p.lm_head, p.V, p.H, x);
    return it;
  }
  const int l = idx / 5;
  const SLayer& Ly = p.L[l];
  it.kind = idx % 5;
  it.layer = l;
  switch (it.kind) {
    case IT_QKV: rows_item(it, Ly.w_qkv, (p.Hq + 2 * p.Hkv) * kD, p.H, x); break;
    case IT_O: rows_item(it, Ly.w_o, p.H, p.Hq * kD, x); break;
    case IT_DOWN: rows_item(it, Ly.w_down, p.H, p.F, x); break;
    case IT_GU: {
      const Span sp = span_of(p.F, x.c, x.n_cta);
      it.row_bytes = p.H * 2;
      it.rps = min(kFlush, kStageB / it.row_bytes);
      it.r0 = sp.r0;
      it.n1 = it.n2 = sp.n;
      it.src1 = (const unsigned char*)(Ly.w_gu + (size_t)sp.r0 * p.H);
      it.src2 = (const unsigned char*)(Ly.w_gu + ((size_t)p.F + sp.r0) * p.H);
      it.n_stages = 2 * ((sp.n + it.rps - 1) / it.rps);
      break;
    }
    default: {  // IT_KV
      const KvSplit k = kv_split(x.c, x.n_cta, p.Hkv, x.len);
      it.g = k.g; it.s = k.s; it.n_split = k.n_split; it.t0 = k.t0; it.t1 = k.t1;
      it.n_stages = k.g < 0 ? 0 : (k.t1 - k.t0 + kTokS - 1) / kTokS;
      break;
    }
  }
  return it;
}

// (item-local first row, rows) of stage k of a rows item
QD_DEV void stage_rows(const Item& it, int k, int& lr0, int& nr, const unsigned char*& src) {
  const int s1 = (it.n1 + it.rps - 1) / it.rps;
  if (k < s1) {
    lr0 = k * it.rps;
    nr = min(it.rps, it.n1 - lr0);
    src = it.src1 + (size_t)lr0 * it.row_bytes;
  } else {
    const int kk = (k - s1) * it.rps;
    lr0 = it.n1 + kk;
    nr = min(it.rps, it.n2 - kk);
    src = it.src2 + (size_t)kk * it.row_bytes;
  }
}

// Cache row of logical token t of kv head g (the tensor maps' row index); -1 when
// the page id is out of range (the caller records the error).
QD_DEV int kv_row(const SParams& p, int g, int t) {
  const PagedSlot sl = paged_slot(p.page_table, t, p.page_size, p.n_pages);
  if (!sl.ok) return -1;
  return (sl.page * p.Hkv + g) * p.page_size + sl.slot;
}

// ---------------------------------------------------------------- producer
struct Cursor {
  int idx, k;
  Item it;
};
QD_DEV void cur_settle(const SParams& p, const Ctx& x, Cursor& c) {
  while (c.it.kind != IT_END && c.k >= c.it.n_stages) {
    ++c.idx;
    c.k = 0;
    c.it = get_item(p, x, c.idx);
  }
}

QD_DEV void issue_stage(const SParams& p, const STmaps& tm, const Ctx& x, const Cursor& c, unsigned char* dst,
                        uint64_t* bar, uint64_t pol) {
  const Item& it = c.it;
  if (it.kind != IT_KV) {
    int lr0, nr;
    const unsigned char* src;
    stage_rows(it, c.k, lr0, nr, src);
    const uint32_t bytes = (uint32_t)nr * (uint32_t)it.row_bytes;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s_hint(dst, src, bytes, bar, pol);
    return;
  }
  // K/V: 16-token boxes of K (two 64-column halves) then V, the current token's
  // granule only up to the token itself (its row comes from the consumers)
  const int ta = it.t0 + c.k * kTokS, tb = min(it.t1, ta + kTokS);
  const int copy_end = min(tb, x.pos);
  int nseg = 0;
  for (int u = ta; u < copy_end; u += 16) ++nseg;
  mbar_arrive_expect_tx(bar, (uint32_t)nseg * 4 * 16 * 128);
  const uint32_t d0 = smem_u32(dst);
  for (int u = ta, k = 0; u < copy_end; u += 16, ++k) {
    int row = kv_row(p, it.g, u);
    if (row < 0) {
      set_error(p.err, QD_DEVERR_PAGE);
      row = 0;
    }
    const uint32_t dk = d0 + k * 16 * 128, dv = dk + kTokS * kD * 2;
    const CUtensorMap* mk = &tm.k[it.layer];
    const CUtensorMap* mv = &tm.v[it.layer];
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dk),
        "l"((uint64_t)mk), "r"(0), "r"(row), "r"(smem_u32(bar))
        : "memory");
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dk + kTokS * 128),
        "l"((uint64_t)mk), "r"(64), "r"(row), "r"(smem_u32(bar))
        : "memory");
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dv),
        "l"((uint64_t)mv), "r"(0), "r"(row), "r"(smem_u32(bar))
        : "memory");
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dv + kTokS * 128),
        "l"((uint64_t)mv), "r"(64), "r"(row), "r"(smem_u32(bar))
        : "memory");
  }
}

// the same bytes into L2 (fire and forget)
QD_DEV void prefetch_stage(const SParams& p, const Ctx& x, const Cursor& c) {
  const Item& it = c.it;
  if (it.kind != IT_KV) {
    int lr0, nr;
    const unsigned char* src;
    stage_rows(it, c.k, lr0, nr, src);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"((uint32_t)nr * it.row_bytes)
                 : "memory");
    return;
  }
  const int ta = it.t0 + c.k * kTokS, tb = min(it.t1, ta + kTokS);
  const int copy_end = min(tb, x.pos);
  const SLayer& Ly = p.L[it.layer];
  for (int u = ta; u < copy_end; u += 16) {
    const int row = kv_row(p, it.g, u);
    if (row < 0) continue;
    // rows of one granule lie in one page (the page size is a multiple of 16, or the
    // cache is one page); stay inside it
    const PagedSlot sl = paged_slot(p.page_table, u, p.page_size, p.n_pages);
    const int nrow = min(16, p.page_size - sl.slot);
    const uint32_t bytes = (uint32_t)nrow * kD * 2;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(Ly.k_cache + (size_t)row * kD), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(Ly.v_cache + (size_t)row * kD), "r"(bytes)
                 : "memory");
  }
}

// The producer runs the L2 read-ahead kPfAhead stages ahead of its copies while
// the stream flows, and up to kPfStall stages ahead while it waits for a free ring
// slot (the consumers are stalled on a dependency): HBM then keeps fetching the
// coming weights into L2, and the ring refills from L2 once the consumers resume.
QD_DEV void producer(const SParams& p, const STmaps& tm, const Ctx& x, const Smem& S, volatile int* s_abort) {
  const uint64_t pol = policy_evict_first();
  Cursor cp, pf;
  cp.idx = pf.idx = 0;
  cp.k = pf.k = 0;
  cp.it = pf.it = get_item(p, x, 0);
  cur_settle(p, x, cp);
  cur_settle(p, x, pf);
  int ahead = 0;  // stages the read-ahead cursor is in front of the copy cursor
  auto pf_step = [&]() {
    prefetch_stage(p, x, pf);
    ++pf.k;
    cur_settle(p, x, pf);
    ++ahead;
  };
  while (ahead < kPfAhead && pf.it.kind != IT_END) pf_step();
  int issued = 0;
  bool ok = true;
  while (cp.it.kind != IT_END) {
    const int slot = issued % kNSt;
    if (issued >= kNSt) {
      uint64_t* bar = &S.empty[slot];
      const uint32_t parity = (uint32_t)(((issued / kNSt) - 1) & 1);
      if (!mbar_try_wait(bar, parity)) {
        const uint64_t t0 = global_ns();
        bool got = false;
        for (int i = 0; i < (1 << 24); ++i) {
          if (mbar_try_wait(bar, parity)) {
            got = true;
            break;
          }
          if (ahead < kPfStall && pf.it.kind != IT_END) pf_step();
          if ((i & 63) == 63 && (*s_abort || global_ns() - t0 > 1000000000ull)) break;
        }
        if (!got) {
          if (!*s_abort) set_error(p.err, QD_DEVERR_TIMEOUT);
          ok = false;
        }
      }
    }
    if (!ok || *s_abort) break;
    if (cp.k == 0) STRACE(512 + cp.idx);
    if (cp.it.kind == IT_KV && cp.k < 4) STRACE(3000 + 10 * cp.it.layer + cp.k);
    issue_stage(p, tm, x, cp, S.ring + (size_t)slot * kStageB, &S.full[slot], pol);
    ++issued;
    ++cp.k;
    cur_settle(p, x, cp);
    if (ahead > 0) {
      --ahead;
    } else if (pf.it.kind != IT_END) {  // the read-ahead fell level: move it along without fetching
      ++pf.k;
      cur_settle(p, x, pf);
    }
    while (ahead < kPfAhead && pf.it.kind != IT_END) pf_step();
  }
  // a CTA never exits with a copy still landing in its shared memory
  for (int i = max(0, issued - kNSt); i < issued; ++i)
    mbar_wait_bounded(&S.full[i % kNSt], (uint32_t)((i / kNSt) & 1), p.err);
}

// ---------------------------------------------------------------- consumers: GEMV
QD_DEV float dot8(const uint4& w, const float* x) {
  float a = bf_lo(w.x) * x[0], b = bf_hi(w.x) * x[1];
  a = fmaf(bf_lo(w.y), x[2], a);
  b = fmaf(bf_hi(w.y), x[3], b);
  a = fmaf(bf_lo(w.z), x[4], a);
  b = fmaf(bf_hi(w.z), x[5], b);
  a = fmaf(bf_lo(w.w), x[6], a);
  b = fmaf(bf_hi(w.w), x[7], b);
  return a + b;
}
QD_DEV float silu(float g) { return g / (1.0f + expf(-g)); }
QD_DEV uint32_t bf16x2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// Consumers: wait until *cnt >= target (thread 0 polls, the others wait at the
// consumer barrier). False on a timeout or an abort, which then ends this CTA too.
QD_DEV bool cwait(const int* cnt, int target, const Smem& S, int* abort_w, int* err, volatile int* s_abort) {
  if (cnt == nullptr) return true;
  if (threadIdx.x == 0) S.misc_i[1] = wait_count(cnt, target, abort_w, err) ? 1 : 0;
  cbar();
  const bool r = S.misc_i[1] != 0;
  if (!r && threadIdx.x == 0) *s_abort = 1;
  return r;
}

enum { P_NORM_RES = 0, P_NORM_EMB = 1, P_BF16 = 2 };
enum { E_STORE = 0, E_RES = 1, E_PAIR = 2, E_LM = 3 };

struct GemvJob {
  const int* wait_cnt;       // dependency: *wait_cnt >= wait_target before the activation is read
  int wait_target;
  int K;
  int pro;
  const __nv_bfloat16* xb;   // P_NORM_EMB: embedding row; P_BF16: activation
  const __nv_bfloat16* nw;   // RMSNorm weight
  int epi;
  float* y;                  // E_STORE / E_LM
  const __nv_bfloat16* emb;  // E_RES: residual base from this embedding row (first layer's O)
  int trace_ev;              // profiling build: the event stamped once the wait is over
};

struct Cand {
  float v;
  int i;
};
QD_DEV bool better(const Cand& a, const Cand& b) { return a.v > b.v || (a.v == b.v && a.i < b.i); }

QD_DEV int c_of(int K) {
  const int ch = K / 8;
  return ch <= kCT ? 1 : ch <= 2 * kCT ? 2 : ch <= 3 * kCT ? 3 : ch <= 4 * kCT ? 4 : 6;
}

// One projection item: prologue, every stage of the item from the ring,
// reduction windows, epilogue. Returns false on an abort.
template <int C>
QD_DEV bool gemv_item(const SParams& p, const Item& it, const GemvJob& J, const Smem& S, int& gs, Cand& best,
                      volatile int* s_abort, int* abort_w) {
  constexpr int RB = C == 1 ? 8 : C == 2 ? 4 : 2;   // rows per register batch
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = J.K;
  const int chunks = K / 8;
  const int T = min(kCT, (((chunks + C - 1) / C) + 31) / 32 * 32);
  const int P = kCT / T;
  const int grp = tid / T, t = tid - grp * T;
  const int wpg = T >> 5, wig = t >> 5;
  const bool in_grp = grp < P;
  int col[C];
  bool cv[C];
#pragma unroll
  for (int j = 0; j < C; ++j) {
    col[j] = (j * T + t) * 8;
    cv[j] = in_grp && col[j] < K;
  }

  // ---- prologue: this thread's activation slice
  float xv[C][8];
#pragma unroll
  for (int j = 0; j < C; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) xv[j][e] = 0.f;
  // the RMSNorm weights do not depend on the earlier phases: load them before the wait
  uint4 wn[C];
#pragma unroll
  for (int j = 0; j < C; ++j)
    wn[j] = (J.pro != P_BF16 && cv[j]) ? *(const uint4*)(J.nw + col[j]) : make_uint4(0u, 0u, 0u, 0u);
  if (!cwait(J.wait_cnt, J.wait_target, S, abort_w, p.err, s_abort)) return false;
  if (tid == 0) STRACE(J.trace_ev);
  if (J.pro == P_BF16) {
#pragma unroll
    for (int j = 0; j < C; ++j) {
      if (!cv[j]) continue;
      const uint4 v = __ldcg((const uint4*)(J.xb + col[j]));
      xv[j][0] = bf_lo(v.x); xv[j][1] = bf_hi(v.x); xv[j][2] = bf_lo(v.y); xv[j][3] = bf_hi(v.y);
      xv[j][4] = bf_lo(v.z); xv[j][5] = bf_hi(v.z); xv[j][6] = bf_lo(v.w); xv[j][7] = bf_hi(v.w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < C; ++j) {
      if (!cv[j]) continue;
      if (J.pro == P_NORM_EMB) {
        const uint4 v = *(const uint4*)(J.xb + col[j]);
        xv[j][0] = bf_lo(v.x); xv[j][1] = bf_hi(v.x); xv[j][2] = bf_lo(v.y); xv[j][3] = bf_hi(v.y);
        xv[j][4] = bf_lo(v.z); xv[j][5] = bf_hi(v.z); xv[j][6] = bf_lo(v.w); xv[j][7] = bf_hi(v.w);
      } else {
        const float4 a = __ldcg((const float4*)(p.res + col[j]));
        const float4 b = __ldcg((const float4*)(p.res + col[j] + 4));
        xv[j][0] = a.x; xv[j][1] = a.y; xv[j][2] = a.z; xv[j][3] = a.w;
        xv[j][4] = b.x; xv[j][5] = b.y; xv[j][6] = b.z; xv[j][7] = b.w;
      }
    }
    float ss = 0.f;
    if (grp == 0) {
#pragma unroll
      for (int j = 0; j < C; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(xv[j][e], xv[j][e], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) S.misc_f[warp] = ss;
    cbar();
    float tot = 0.f;
    for (int w = 0; w < wpg; ++w) tot += S.misc_f[w];
    const float inv = 1.0f / sqrtf(tot / (float)K + p.eps);
#pragma unroll
    for (int j = 0; j < C; ++j) {
      const float nw[8] = {bf_lo(wn[j].x), bf_hi(wn[j].x), bf_lo(wn[j].y), bf_hi(wn[j].y),
                           bf_lo(wn[j].z), bf_hi(wn[j].z), bf_lo(wn[j].w), bf_hi(wn[j].w)};
#pragma unroll
      for (int e = 0; e < 8; ++e) xv[j][e] = cv[j] ? round_bf16(nw[e] * round_bf16(xv[j][e] * inv)) : 0.f;
    }
    // (misc_f is written again only after the flush barriers that end this item)
  }

  // ---- reduction windows
  auto epilogue = [&](int lr, float s) {
    if (J.epi == E_STORE) {
      J.y[it.r0 + lr] = s;
    } else if (J.epi == E_RES) {  // this CTA owns these rows of the residual: its copy is in smem
      const int r = it.r0 + lr;
      const float v = (J.emb ? __bfloat162float(J.emb[r]) : S.resown[lr]) + s;
      p.res[r] = v;
      S.resown[lr] = v;
    } else if (J.epi == E_PAIR) {
      S.pair[lr] = s;
    } else {
      const int r = it.r0 + lr;
      J.y[r] = s;
      const Cand d{isnan(s) ? -INFINITY : s, isnan(s) ? INT_MAX : r};
      if (better(d, best)) best = d;
    }
  };
  auto flush = [&](int base, int nrows) {
    cbar();
    for (int r = tid; r < nrows; r += kCT) {
      float s = 0.f;
      for (int k = 0; k < wpg; ++k) s += S.red[r * wpg + k];
      epilogue(base + r, s);
    }
    cbar();
  };

  int wbase = 0;  // first item-local row of the current window
  for (int k = 0; k < it.n_stages; ++k) {
    int lr0, nr;
    const unsigned char* src_unused;
    stage_rows(it, k, lr0, nr, src_unused);
    if (lr0 + nr - wbase > kFlush) {
      flush(wbase, lr0 - wbase);
      wbase = lr0;
    }
    const int slot = gs % kNSt;
    const bool got = mbar_wait_bounded(&S.full[slot], (uint32_t)((gs / kNSt) & 1), p.err);
    if (!cbar_and(got)) {
      if (tid == 0) *s_abort = 1;
      return false;
    }
    if (k == 0 && tid == 0) STRACE(1024 + J.trace_ev);
    const unsigned char* st = S.ring + (size_t)slot * kStageB;
    if (in_grp) {
      for (int b0 = 0; b0 < nr; b0 += P * RB) {
        uint4 w[RB][C];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int rr = b0 + grp + P * u;
#pragma unroll
          for (int j = 0; j < C; ++j)
            w[u][j] = (rr < nr && cv[j]) ? *(const uint4*)(st + (size_t)rr * it.row_bytes + (size_t)col[j] * 2)
                                        : make_uint4(0u, 0u, 0u, 0u);
        }
        float v[RB];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          float a = 0.f;
#pragma unroll
          for (int j = 0; j < C; ++j) a += dot8(w[u][j], xv[j]);
          v[u] = a;
        }
        // transposed butterfly: lane l ends with the warp sum of row rsel(l)
        int rsel = 0;
#pragma unroll
        for (int L = 16, n = RB; L >= 1; L >>= 1) {
          if (n > 1) {
            const int hh = n / 2;
            const bool up = (lane & L) != 0;
#pragma unroll
            for (int q = 0; q < hh; ++q) {
              const float send = up ? v[q] : v[q + hh];
              const float keep = up ? v[q + hh] : v[q];
              v[q] = keep + __shfl_xor_sync(0xffffffffu, send, L);
            }
            if (up) rsel += hh;
            n = hh;
          } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], L);
          }
        }
        constexpr int kLow = 32 / RB - 1;
        const int rr = b0 + grp + P * rsel;
        if ((lane & kLow) == 0 && rr < nr) S.red[(lr0 + rr - wbase) * wpg + wig] = v[0];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);
    ++gs;
  }
  if (tid == 0) STRACE(1536 + J.trace_ev);
  flush(wbase, it.n1 + it.n2 - wbase);
  if (J.epi == E_PAIR) {  // h = bf16(silu(gate) * up) of this CTA's pairs
    for (int j = tid; j < it.n1; j += kCT)
      p.h[it.r0 + j] = __float2bfloat16_rn(silu(S.pair[j]) * S.pair[it.n1 + j]);
  }
  return true;
}

QD_DEV bool run_gemv(const SParams& p, const Item& it, const GemvJob& J, const Smem& S, int& gs, Cand& best,
                     volatile int* s_abort, int* abort_w) {
  switch (c_of(J.K)) {
    case 1: return gemv_item<1>(p, it, J, S, gs, best, s_abort, abort_w);
    case 2: return gemv_item<2>(p, it, J, S, gs, best, s_abort, abort_w);
    case 3: return gemv_item<3>(p, it, J, S, gs, best, s_abort, abort_w);
    case 4: return gemv_item<4>(p, it, J, S, gs, best, s_abort, abort_w);
    default: return gemv_item<6>(p, it, J, S, gs, best, s_abort, abort_w);
  }
}

// ---------------------------------------------------------------- consumers: attention
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
// byte offset of (row r, 16-byte chunk c) in a K or V tile of the stage: each
// 64-column half of the rows is its own [kTokS x 128 B] block in the 128-byte
// swizzle the copy engine writes (chunk c of row r at c ^ (r & 7))
QD_DEV uint32_t swz(int r, int c) {
  return (uint32_t)((c >> 3) * (kTokS * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// This CTA's attention split of layer l: QK-norm + RoPE of q (and of the new k,
// v if the current token is in this split, which then goes to the cache), the
// split's K/V tiles from the ring on the tensor cores, the split's partial and
// the ticket; the last split of the kv head combines all partials in split order.
QD_DEV bool attn_item(const SParams& p, const Item& it, const Smem& S, int& gs, int pos, int len,
                      volatile int* s_abort, int* abort_w) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int REP = p.rep;
  const int g = it.g;
  const SLayer& Ly = p.L[it.layer];
  const bool own_pos = pos >= it.t0 && pos < it.t1;
  // ---- q (pre-scaled by scale * log2 e) as bf16 hi + lo, heads padded to 8; new k, v.
  // One warp per head vector (lane l holds dims 4l .. 4l + 3): the RMSNorm is a warp
  // reduction and RoPE's partner dim d ^ 64 sits in lane l ^ 16, so no CTA barrier is
  // needed until the vectors are in shared memory.
  float* s_knew = S.obuf;          // [128] bf16-valued new k (the split holding pos)
  float* s_vnew = S.obuf + kD;     // [128] new v
  {
    const int d0 = lane * 4;
    // the RoPE row and the QK-norm weights do not depend on the projection: load
    // them before waiting for it
    const float4 c01 = *(const float4*)(p.rope + (size_t)pos * (kD / 2) + (d0 & 63));
    const float4 c23 = *(const float4*)(p.rope + (size_t)pos * (kD / 2) + (d0 & 63) + 2);
    const float cs_c[4] = {c01.x, c01.z, c23.x, c23.z}, cs_s[4] = {c01.y, c01.w, c23.y, c23.w};
    const uint2 wqb = *(const uint2*)(Ly.q_norm + d0), wkb = *(const uint2*)(Ly.k_norm + d0);
    const float wq[4] = {bf_lo(wqb.x), bf_hi(wqb.x), bf_lo(wqb.y), bf_hi(wqb.y)};
    const float wk[4] = {bf_lo(wkb.x), bf_hi(wkb.x), bf_lo(wkb.y), bf_hi(wkb.y)};
    for (int e = tid; e < (kHP - REP) * kD; e += kCT) {  // padded heads stay zero
      S.qh[REP * kD + e] = __float2bfloat16_rn(0.f);
      S.ql[REP * kD + e] = __float2bfloat16_rn(0.f);
    }
    if (!cwait(p.sync + 5 * it.layer + PH_QKV, gridDim.x, S, abort_w, p.err, s_abort)) return false;
    if (tid == 0) STRACE(10 * it.layer + 2);
    for (int i = warp; i <= REP; i += kCW) {
      if (i == REP && !own_pos) break;
      const int row = i < REP ? (g * REP + i) : (p.Hq + g);
      const float4 xv4 = __ldcg((const float4*)(p.qkv + (size_t)row * kD + d0));
      float4 vv4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i == REP) vv4 = __ldcg((const float4*)(p.qkv + (size_t)(p.Hq + p.Hkv + g) * kD + d0));
      const float x[4] = {xv4.x, xv4.y, xv4.z, xv4.w};
      const float inv = 1.0f / sqrtf(warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]) / (float)kD + p.eps);
      float y[4], r[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) y[e] = round_bf16((i < REP ? wq[e] : wk[e]) * round_bf16(x[e] * inv));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, y[e], 16);
        r[e] = (d0 < 64) ? (y[e] * cs_c[e] - other * cs_s[e]) : (y[e] * cs_c[e] + other * cs_s[e]);
      }
      if (i < REP) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float qv = r[e] * p.scale_log2;
          const __nv_bfloat16 hi = __float2bfloat16_rn(qv);
          S.qh[i * kD + d0 + e] = hi;
          S.ql[i * kD + d0 + e] = __float2bfloat16_rn(qv - __bfloat162float(hi));
        }
      } else {  // the current token's k (normed, rotated) and v: to the cache and to smem
        const float vx[4] = {vv4.x, vv4.y, vv4.z, vv4.w};
        __nv_bfloat16 kb[4], vb[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          kb[e] = __float2bfloat16_rn(r[e]);
          vb[e] = __float2bfloat16_rn(vx[e]);
          s_knew[d0 + e] = __bfloat162float(kb[e]);
          s_vnew[d0 + e] = __bfloat162float(vb[e]);
        }
        const int crow = kv_row(p, g, pos);
        if (crow < 0) {
          if (lane == 0) set_error(p.err, QD_DEVERR_PAGE);
        } else {
          *(uint2*)(Ly.k_cache + (size_t)crow * kD + d0) =
              make_uint2(bf16x2(kb[0], kb[1]), bf16x2(kb[2], kb[3]));
          *(uint2*)(Ly.v_cache + (size_t)crow * kD + d0) =
              make_uint2(bf16x2(vb[0], vb[1]), bf16x2(vb[2], vb[3]));
        }
      }
    }
    cbar();
  }
  if (tid == 0) STRACE(2048 + 10 * it.layer + 0);
  // B fragments of Q^T for the 8 k-steps: head n = lane / 4, dims 16 ks + 2 (lane % 4) (+ 8)
  const int qn = lane >> 2, qk = (lane & 3) * 2;
  uint32_t qh[8][2], ql[8][2];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    qh[ks][0] = *(const uint32_t*)(S.qh + qn * kD + ks * 16 + qk);
    qh[ks][1] = *(const uint32_t*)(S.qh + qn * kD + ks * 16 + qk + 8);
    ql[ks][0] = *(const uint32_t*)(S.ql + qn * kD + ks * 16 + qk);
    ql[ks][1] = *(const uint32_t*)(S.ql + qn * kD + ks * 16 + qk + 8);
  }
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
  const int rA = (lane & 7) + ((lane >> 3) & 1) * 8, cA = lane >> 4;
  const int rV = (lane & 7) + ((lane >> 4) & 1) * 8, cV = (lane >> 3) & 1;
  __nv_bfloat16* sPh = S.pb + warp * 2 * kHP * 16;
  __nv_bfloat16* sPl = sPh + kHP * 16;

  for (int k = 0; k < it.n_stages; ++k) {
    const int ta = it.t0 + k * kTokS, tb = min(it.t1, ta + kTokS);
    const int nv = tb - ta;
    const int slot = gs % kNSt;
    const bool got = mbar_wait_bounded(&S.full[slot], (uint32_t)((gs / kNSt) & 1), p.err);
    if (!cbar_and(got)) {
      if (tid == 0) *s_abort = 1;
      return false;
    }
    if (k == 0 && tid == 0) STRACE(2048 + 10 * it.layer + 1);
    if (k < 4 && tid == 0) STRACE(3400 + 10 * it.layer + k);
    unsigned char* st = S.ring + (size_t)slot * kStageB;
    const uint32_t sK = smem_u32(st), sV = sK + kTokS * kD * 2;
    // rows past the split hold any bits: zero their V (their scores are masked);
    // the current token's row comes from registers
    bool wrote = false;
    if (nv < kTokS) {
      for (int e = tid; e < (kTokS - nv) * 16; e += kCT) {
        const int r = nv + (e >> 4), c = e & 15;
        *(uint4*)(st + kTokS * kD * 2 + swz(r, c)) = make_uint4(0u, 0u, 0u, 0u);
      }
      wrote = true;
    }
    if (own_pos && pos >= ta && pos < tb) {
      if (tid < kD) {
        const int r = pos - ta;
        const uint32_t o16 = swz(r, tid >> 3) + (uint32_t)((tid & 7) * 2);
        *(__nv_bfloat16*)(st + o16) = __float2bfloat16_rn(s_knew[tid]);
        *(__nv_bfloat16*)(st + kTokS * kD * 2 + o16) = __float2bfloat16_rn(s_vnew[tid]);
      }
      wrote = true;
    }
    if (wrote) {
      fence_proxy_async_smem();  // these generic writes come before the slot's next copy
      cbar();
    }
    if (warp * 16 < nv) {
      // ---- S^T = K . Q^T for this warp's 16 tokens
      uint32_t a[8][4];
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) ldsm_x4(a[ks], sK + swz(warp * 16 + rA, 2 * ks + cA));
      float sc[4][4] = {};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        mma16816(sc[ks & 1], a[ks], qh[ks][0], qh[ks][1]);
        mma16816(sc[2 + (ks & 1)], a[ks], ql[ks][0], ql[ks][1]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[0][e] = (sc[0][e] + sc[1][e]) + (sc[2][e] + sc[3][e]);
      float* scr = sc[0];
      const int tr0 = ta + warp * 16 + (lane >> 2), tr1 = tr0 + 8;
      if (tr0 >= tb) { scr[0] = -INFINITY; scr[1] = -INFINITY; }
      if (tr1 >= tb) { scr[2] = -INFINITY; scr[3] = -INFINITY; }
      // ---- online softmax over this warp's tokens
      float mx0 = fmaxf(scr[0], scr[2]), mx1 = fmaxf(scr[1], scr[3]);
#pragma unroll
      for (int o2 = 4; o2 <= 16; o2 <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
      const float al1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
      const float p00 = scr[0] == -INFINITY ? 0.f : exp2f(scr[0] - mn0);
      const float p01 = scr[1] == -INFINITY ? 0.f : exp2f(scr[1] - mn1);
      const float p10 = scr[2] == -INFINITY ? 0.f : exp2f(scr[2] - mn0);
      const float p11 = scr[3] == -INFINITY ? 0.f : exp2f(scr[3] - mn1);
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
      // ---- O^T += V^T . P^T, 8 tiles of 16 dims
      uint32_t av[8][4];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) ldsm_x4_t(av[mt], sV + swz(warp * 16 + rV, 2 * mt + cV));
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        mma16816(o[mt], av[mt], pb0h, pb1h);
        mma16816(o[mt], av[mt], pb0l, pb1l);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);
    ++gs;
  }

  if (tid == 0) STRACE(2048 + 10 * it.layer + 2);
  // ---- merge the warps (heads in chunks of 4) into the split's partial
  const size_t slot0 = (size_t)g * kMaxSplit;
  const size_t sslot = slot0 + it.s;
  {
    const int h0 = (lane & 3) * 2;
    if (lane < 4) {
      S.sM[warp * kHP + h0] = m0;
      S.sM[warp * kHP + h0 + 1] = m1;
      S.sL[warp * kHP + h0] = l0;
      S.sL[warp * kHP + h0 + 1] = l1;
    }
  }
  for (int hc = 0; hc < REP; hc += 4) {
    const int h0 = (lane & 3) * 2, d0 = lane >> 2;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int hh = h0 + e - hc;
      if (hh >= 0 && hh < 4) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          S.obuf[(warp * 4 + hh) * kD + mt * 16 + d0] = o[mt][e];
          S.obuf[(warp * 4 + hh) * kD + mt * 16 + d0 + 8] = o[mt][2 + e];
        }
      }
    }
    cbar();
    for (int e = tid; e < 4 * kD; e += kCT) {
      const int hh = e / kD, d = e % kD, h = hc + hh;
      if (h >= REP) continue;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kCW; ++w) M = fmaxf(M, S.sM[w * kHP + h]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < kCW; ++w) {
        const float c = S.sM[w * kHP + h] == -INFINITY ? 0.f : exp2f(S.sM[w * kHP + h] - M);
        L = fmaf(c, S.sL[w * kHP + h], L);
        O = fmaf(c, S.obuf[(w * 4 + hh) * kD + d], O);
      }
      p.part[(sslot * REP + h) * kD + d] = O;
      if (d == 0) {
        p.part_ml[(sslot * REP + h) * 2 + 0] = M;
        p.part_ml[(sslot * REP + h) * 2 + 1] = L;
      }
    }
    cbar();
  }
  int* tickets = p.sync + 5 * p.n_layers;
  if (tid == 0) STRACE(2048 + 10 * it.layer + 3);
  if (tid == 0) S.misc_i[0] = atom_acq_rel_add(tickets + g, 1);
  cbar();
  if (tid == 0) STRACE(2048 + 10 * it.layer + 4);
  if (S.misc_i[0] != it.n_split - 1) return true;
  // ---- the last split combines: (max, sum) of every split staged together, the
  // weights exp2(m_k - M) per head, then each output element from all splits' partials
  // with the loads in flight together
  float* sMk = S.red;                      // [n_split][REP] maxima -> weights
  float* sLk = S.red + kMaxSplit * 8;      // [n_split][REP] sums
  float* sTot = S.pair;                    // [REP] totals
  for (int e = tid; e < it.n_split * REP; e += kCT) {
    const float2 ml = __ldcg((const float2*)(p.part_ml + (slot0 * REP + e) * 2));
    sMk[e] = ml.x;
    sLk[e] = ml.y;
  }
  cbar();
  if (tid == 0) STRACE(2048 + 10 * it.layer + 5);
  if (tid < REP) {
    float M = -INFINITY;
    for (int k = 0; k < it.n_split; ++k) M = fmaxf(M, sMk[k * REP + tid]);
    float L = 0.f;
    for (int k = 0; k < it.n_split; ++k) {
      const float m = sMk[k * REP + tid];
      const float w = m == -INFINITY ? 0.f : exp2f(m - M);
      L = fmaf(w, sLk[k * REP + tid], L);
      sMk[k * REP + tid] = w;
    }
    sTot[tid] = L;
  }
  cbar();
  {
    constexpr int kE = kHP * kD / kCT;   // at most 4 output elements per thread
    const int ne = REP * kD;
    float O[kE];
#pragma unroll
    for (int j = 0; j < kE; ++j) O[j] = 0.f;
    for (int k0 = 0; k0 < it.n_split; k0 += 8) {
      float a[kE][8];
#pragma unroll
      for (int j = 0; j < kE; ++j) {
        const int e = tid + j * kCT;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          a[j][u] = (e < ne && k0 + u < it.n_split)
                        ? __ldcg(p.part + ((slot0 + k0 + u) * REP + e / kD) * kD + (e % kD)) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kE; ++j) {
        const int e = tid + j * kCT;
        if (e >= ne) continue;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (k0 + u < it.n_split) O[j] = fmaf(sMk[(k0 + u) * REP + e / kD], a[j][u], O[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < kE; ++j) {
      const int e = tid + j * kCT;
      if (e < ne) p.attn[(size_t)g * REP * kD + e] = __float2bfloat16_rn(O[j] / sTot[e / kD]);
    }
  }
  cbar();
  if (tid == 0) STRACE(2048 + 10 * it.layer + 6);
  if (tid == 0) {
    tickets[g] = 0;
    red_release_add(p.sync + 5 * it.layer + PH_ATTN, 1);
  }
  return true;
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kST, 1)
    stream_step_kernel(const __grid_constant__ SParams p, const __grid_constant__ STmaps tm) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Smem S;
  S.ring = base + Carve::ring;
  S.full = (uint64_t*)(base + Carve::bars);
  S.empty = S.full + kNSt;
  S.red = (float*)(base + Carve::red);
  S.pair = (float*)(base + Carve::pair);
  S.misc_f = (float*)(base + Carve::misc);
  S.misc_i = (int*)(base + Carve::misc + 64);
  S.qh = (__nv_bfloat16*)(base + Carve::qh);
  S.ql = (__nv_bfloat16*)(base + Carve::ql);
  S.pb = (__nv_bfloat16*)(base + Carve::pbuf);
  S.sM = (float*)(base + Carve::ml);
  S.sL = S.sM + kCW * kHP;
  S.ared = (float*)(base + Carve::ared);
  S.sx = S.ared + 64;
  S.obuf = (float*)(base + Carve::obuf);
  S.resown = (float*)(base + Carve::resown);
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = p.n_layers;
  int* abort_w = p.sync + 5 * L + 65;
  if (tid == 0) {
    for (int i = 0; i < kNSt; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kCW);
    }
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();

  if (tid == 0) STRACE(4095);
  Ctx x;
  x.c = blockIdx.x;
  x.n_cta = gridDim.x;
  x.pos = p.pos[0];
  x.len = x.pos + 1;
  const int cap = p.max_pages * p.page_size;
  if (x.pos < 0 || x.pos >= cap || x.pos >= p.rope_max_pos) {
    if (blockIdx.x == 0 && tid == 0) set_error(p.err, QD_DEVERR_POS);
    return;
  }

  if (warp == kCW) {  // ---- producer warp
    if (lane == 0) producer(p, tm, x, S, &s_abort);
    return;
  }

  // ---- consumer warps
  int tok = p.tok[0];
  if (tok < 0 || tok >= p.V) {
    if (blockIdx.x == 0 && tid == 0) set_error(p.err, QD_DEVERR_PAGE);
    tok = 0;
  }
  const __nv_bfloat16* emb_row = p.embed + (size_t)tok * p.H;
  int gs = 0;
  Cand best{-INFINITY, INT_MAX};
  bool ok = true;
  auto arrive = [&](int* cnt) {  // the phase's stores are ordered before the count
    cbar();
    if (tid == 0) red_release_add(cnt, 1);
  };
  const int n = gridDim.x;
  for (int l = 0; l < L && ok; ++l) {
    const SLayer& Ly = p.L[l];
    int* cnt = p.sync + 5 * l;
    // QKV projection of RMSNorm(res; ln_in) (the embedding row in the first layer)
    {
      const Item it = get_item(p, x, 5 * l + IT_QKV);
      GemvJob J = {};
      J.wait_cnt = l > 0 ? p.sync + 5 * (l - 1) + PH_DOWN : nullptr;
      J.wait_target = n;
      J.trace_ev = 10 * l + 0;
      J.K = p.H; J.pro = l == 0 ? P_NORM_EMB : P_NORM_RES; J.xb = emb_row; J.nw = Ly.ln_in;
      J.epi = E_STORE; J.y = p.qkv;
      ok = run_gemv(p, it, J, S, gs, best, &s_abort, abort_w);
      if (!ok) break;
      arrive(cnt + PH_QKV);
      if (tid == 0) STRACE(10 * l + 1);
    }
    // attention split (+ combine)
    {
      const Item it = get_item(p, x, 5 * l + IT_KV);
      if (it.g >= 0) {
        ok = attn_item(p, it, S, gs, x.pos, x.len, &s_abort, abort_w);
        if (!ok) break;
        if (tid == 0) STRACE(10 * l + 3);
      }
    }
    // O projection + residual (the residual starts as the embedding row)
    {
      const Item it = get_item(p, x, 5 * l + IT_O);
      GemvJob J = {};
      J.wait_cnt = cnt + PH_ATTN;
      J.wait_target = p.Hkv;
      J.trace_ev = 10 * l + 4;
      J.K = p.Hq * kD; J.pro = P_BF16; J.xb = p.attn; J.epi = E_RES; J.emb = l == 0 ? emb_row : nullptr;
      ok = run_gemv(p, it, J, S, gs, best, &s_abort, abort_w);
      if (!ok) break;
      arrive(cnt + PH_O);
      if (tid == 0) STRACE(10 * l + 5);
    }
    // gate+up projection of RMSNorm(res; ln_post), SwiGLU of the pairs
    {
      const Item it = get_item(p, x, 5 * l + IT_GU);
      GemvJob J = {};
      J.wait_cnt = cnt + PH_O;
      J.wait_target = n;
      J.trace_ev = 10 * l + 6;
      J.K = p.H; J.pro = P_NORM_RES; J.nw = Ly.ln_post; J.epi = E_PAIR;
      ok = run_gemv(p, it, J, S, gs, best, &s_abort, abort_w);
      if (!ok) break;
      arrive(cnt + PH_GU);
      if (tid == 0) STRACE(10 * l + 7);
    }
    // down projection + residual
    {
      const Item it = get_item(p, x, 5 * l + IT_DOWN);
      GemvJob J = {};
      J.wait_cnt = cnt + PH_GU;
      J.wait_target = n;
      J.trace_ev = 10 * l + 8;
      J.K = p.F; J.pro = P_BF16; J.xb = p.h; J.epi = E_RES;
      ok = run_gemv(p, it, J, S, gs, best, &s_abort, abort_w);
      if (!ok) break;
      arrive(cnt + PH_DOWN);
      if (tid == 0) STRACE(10 * l + 9);
    }
  }
  if (!ok) return;
  // ---- final RMSNorm + LM head with a running argmax
  {
    const Item it = get_item(p, x, 5 * L);
    GemvJob J = {};
    J.wait_cnt = p.sync + 5 * (L - 1) + PH_DOWN;
    J.wait_target = n;
    J.trace_ev = 10 * L + 0;
    J.K = p.H; J.pro = P_NORM_RES; J.nw = p.final_norm; J.epi = E_LM; J.y = p.logits;
    if (!run_gemv(p, it, J, S, gs, best, &s_abort, abort_w)) return;
  }
  if (tid == 0) STRACE(10 * L + 1);
  // CTA argmax (lowest index among equal maxima), candidate, ticket
  Cand c = best;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Cand d;
    d.v = __shfl_xor_sync(0xffffffffu, c.v, o);
    d.i = __shfl_xor_sync(0xffffffffu, c.i, o);
    if (better(d, c)) c = d;
  }
  float* cv = S.misc_f;
  int* ci = S.misc_i + 4;
  if (lane == 0) {
    cv[warp] = c.v;
    ci[warp] = c.i;
  }
  int* am_ticket = p.sync + 5 * L + 64;
  cbar();
  if (tid == 0) {
    Cand b = {cv[0], ci[0]};
    for (int w = 1; w < kCW; ++w) {
      const Cand d = {cv[w], ci[w]};
      if (better(d, b)) b = d;
    }
    p.cand_v[blockIdx.x] = b.v;
    p.cand_i[blockIdx.x] = b.i;
    __threadfence();
    S.misc_i[2] = atomicAdd(am_ticket, 1);
  }
  cbar();
  if (S.misc_i[2] != n - 1) return;
  __threadfence();
  // the last CTA: the step's token, and the counters back to zero for the next launch
  Cand b{-INFINITY, INT_MAX};
  for (int k = tid; k < n; k += kCT) {
    const Cand d{__ldcg(p.cand_v + k), __ldcg(p.cand_i + k)};
    if (better(d, b)) b = d;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Cand d;
    d.v = __shfl_xor_sync(0xffffffffu, b.v, o);
    d.i = __shfl_xor_sync(0xffffffffu, b.i, o);
    if (better(d, b)) b = d;
  }
  cbar();
  if (lane == 0) {
    cv[warp] = b.v;
    ci[warp] = b.i;
  }
  cbar();
  if (tid == 0) {
    Cand t = {cv[0], ci[0]};
    for (int w = 1; w < kCW; ++w) {
      const Cand d = {cv[w], ci[w]};
      if (better(d, t)) t = d;
    }
    int tk = t.i;
    if (tk == INT_MAX) {
      set_error(p.err, QD_DEVERR_NAN);
      tk = 0;
    }
    const int st = p.step[0];
    if (st >= 0 && st < p.max_steps) p.out_tokens[st] = tk;
    else set_error(p.err, QD_DEVERR_STEPS);
    p.tok[0] = tk;
    p.pos[0] = x.pos + 1;
    p.step[0] = st + 1;
  }
  for (int i = tid; i < 5 * L; i += kCT) p.sync[i] = 0;
  if (tid == 0) *am_ticket = 0;
}

// ---------------------------------------------------------------- host
// Tensor maps of the layer caches, encoded once per (pointer, rows) and reused.
struct MapCache {
  const void* ptr[2 * kStreamMaxLayers] = {};
  uint64_t rows[2 * kStreamMaxLayers] = {};
  CUtensorMap map[2 * kStreamMaxLayers];
};

}  // namespace

size_t stream_ws_bytes(int n_layers, int Hq, int Hkv) {
  const int rep = Hq / Hkv;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al((size_t)Hkv * kMaxSplit * rep * kD * 4) + al((size_t)Hkv * kMaxSplit * rep * 2 * 4) +
         al((size_t)(5 * n_layers + 66) * 4) + 2 * al(1024 * 4);
}

bool stream_step_supported(const StreamStepArgs& a) {
  if (a.n_layers < 1 || a.n_layers > kStreamMaxLayers) return false;
  const int rep = a.Hq / a.Hkv;
  if (a.Hq % a.Hkv || !(rep == 1 || rep == 2 || rep == 4 || rep == 8)) return false;
  if (a.Hkv > 64 || a.Hkv > dev_info().sm_count) return false;
  const int ks[3] = {a.H, a.Hq * kD, a.F};
  for (int K : ks)
    if (K < 8 || K % 8 || K / 8 > 6 * kCT || K * 2 > kStageB) return false;
  // gate/up pairs and residual rows per CTA fit their buffers
  if ((a.F + dev_info().sm_count - 1) / dev_info().sm_count > kMaxPair) return false;
  if ((a.H + dev_info().sm_count - 1) / dev_info().sm_count > kMaxOwnRows) return false;
  // 16-token granules never cross a page
  if (!(a.max_pages == 1 || a.page_size % 16 == 0)) return false;
  if (dev_info().max_smem_optin < (int)kSmemBytes) return false;
  return true;
}

cudaError_t launch_stream_step(const StreamStepArgs& a, const Launch& Lh) {
  static SParams p;  // host staging of the launch parameters (copied at launch)
  static STmaps tm;
  static MapCache cache;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  memset(&p, 0, sizeof(p));
  const uint64_t rows = (uint64_t)a.n_pages * a.Hkv * a.page_size;
  for (int l = 0; l < a.n_layers; ++l) {
    const StreamLayerPtrs& s = a.layers[l];
    p.L[l].w_qkv = (const __nv_bfloat16*)s.w_qkv;
    p.L[l].w_o = (const __nv_bfloat16*)s.w_o;
    p.L[l].w_gu = (const __nv_bfloat16*)s.w_gu;
    p.L[l].w_down = (const __nv_bfloat16*)s.w_down;
    p.L[l].ln_in = (const __nv_bfloat16*)s.ln_in;
    p.L[l].ln_post = (const __nv_bfloat16*)s.ln_post;
    p.L[l].q_norm = (const __nv_bfloat16*)s.q_norm;
    p.L[l].k_norm = (const __nv_bfloat16*)s.k_norm;
    p.L[l].k_cache = (__nv_bfloat16*)s.k_cache;
    p.L[l].v_cache = (__nv_bfloat16*)s.v_cache;
    const void* ptrs[2] = {s.k_cache, s.v_cache};
    for (int kv = 0; kv < 2; ++kv) {
      const int i = 2 * l + kv;
      if (cache.ptr[i] != ptrs[kv] || cache.rows[i] != rows) {
        cudaError_t e = encode_tmap_bf16_2d(&cache.map[i], ptrs[kv], rows, kD, 16);
        if (e != cudaSuccess) {
          cache.ptr[i] = nullptr;
          return e;
        }
        cache.ptr[i] = ptrs[kv];
        cache.rows[i] = rows;
      }
      if (kv == 0) tm.k[l] = cache.map[i];
      else tm.v[l] = cache.map[i];
    }
  }
  p.n_layers = a.n_layers;
  p.H = a.H; p.Hq = a.Hq; p.Hkv = a.Hkv; p.F = a.F; p.V = a.V; p.rep = a.Hq / a.Hkv;
  p.eps = a.eps;
  p.scale_log2 = (1.0f / sqrtf((float)kD)) * kLog2e;
  p.embed = (const __nv_bfloat16*)a.embed;
  p.final_norm = (const __nv_bfloat16*)a.final_norm;
  p.lm_head = (const __nv_bfloat16*)a.lm_head;
  p.page_table = a.page_table;
  p.page_size = a.page_size; p.max_pages = a.max_pages; p.n_pages = a.n_pages;
  p.rope = (const float2*)a.rope;
  p.rope_max_pos = a.rope_max_pos;
  p.tok = a.tok; p.pos = a.pos; p.step = a.step; p.out_tokens = a.out_tokens; p.max_steps = a.max_steps;
  p.logits = a.logits;
  p.res = a.res; p.qkv = a.qkv; p.attn = (__nv_bfloat16*)a.attn; p.h = (__nv_bfloat16*)a.h;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  unsigned char* w = (unsigned char*)a.ws;
  const int rep = a.Hq / a.Hkv;
  p.part = (float*)w;
  w += al((size_t)a.Hkv * kMaxSplit * rep * kD * 4);
  p.part_ml = (float*)w;
  w += al((size_t)a.Hkv * kMaxSplit * rep * 2 * 4);
  p.sync = (int*)w;
  w += al((size_t)(5 * a.n_layers + 66) * 4);
  p.cand_v = (float*)w;
  w += al(1024 * 4);
  p.cand_i = (int*)w;
  p.err = Lh.err;

  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(stream_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = std::min(dev_info().sm_count, 1024);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kST);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = Lh.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stream_step_kernel, p, tm);
}

#ifdef QD_STREAM_TRACE
extern "C" int qd_stream_trace_set(void* buf) {
  unsigned long long* p = (unsigned long long*)buf;
  return cudaMemcpyToSymbol(g_stream_trace, &p, sizeof(p)) == cudaSuccess ? 0 : -3;
}
#endif

}  // namespace qd
