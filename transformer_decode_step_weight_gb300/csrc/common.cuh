// Shared device helpers for the sm_103a decode kernels: streaming loads,
// programmatic-dependent-launch controls, bf16 widening, reductions.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "qd.h"
#include "kernels.h"

#define QD_DEV __device__ __forceinline__

namespace qd {

// L2 policy for data read exactly once (weights, KV): evict first, so streamed
// bytes do not push the small re-used activations out of L2.
QD_DEV uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// L2 policies for data kept until a later kernel reads it (evict_last) or for
// the default priority (evict_normal).
QD_DEV uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
QD_DEV uint64_t policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 128-bit streaming load through the non-coherent path without L1 allocation.
QD_DEV uint4 ld_stream(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
QD_DEV uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Programmatic dependent launch. wait(): block until the grids this launch
// depends on have completed and their memory is visible. Every kernel calls it
// before touching memory written by an earlier kernel of the step, and before
// its own first global write. launch_dependents(): allow the next kernel in
// the stream to be scheduled now (it still waits before reading our results).
QD_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
QD_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// bf16 pair (packed in a 32-bit word, low half first) -> two floats, exactly.
QD_DEV float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
QD_DEV float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// binary32 -> bf16 bits, round to nearest even (finite inputs).
QD_DEV uint32_t f2bf_bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}
QD_DEV float round_bf16(float f) { return __uint_as_float(f2bf_bits(f) << 16); }

QD_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
QD_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Physical place of logical token t of a sequence in a paged K/V cache: the
// page-table row pt_row names the page of logical page t / ps, and the token
// sits in slot t % ps of it. Every kernel that reads or writes the cache through
// a page table, and the test export of the gather indices, go through this
// function. A page id outside [0, n_pages) is not followed: ok is false and the
// page is 0 (callers set QD_DEVERR_PAGE).
struct PagedSlot {
  int page, slot;
  bool ok;
};
QD_DEV PagedSlot paged_slot(const int32_t* pt_row, int t, int ps, int n_pages) {
  const int lp = t / ps;
  const int page = pt_row[lp];
  const bool ok = page >= 0 && page < n_pages;
  return PagedSlot{ok ? page : 0, t - lp * ps, ok};
}

// Sticky device error word (bits QD_DEVERR_*), one per process.
QD_DEV void set_error(int* err, int bit) {
  if (err) atomicOr(err, bit);
}

}  // namespace qd

// ---------------------------------------------------------------------------
// Asynchronous bulk copies (TMA, non-tensor form) completing on an mbarrier.
namespace qd {

QD_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

QD_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
QD_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

QD_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

QD_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

QD_DEV bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}

QD_DEV uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for `phase` of the barrier to complete, giving up after limit_ns
// nanoseconds (or 2^24 polls; sets QD_DEVERR_TIMEOUT = 16 and returns false).
// Never unbounded.
QD_DEV bool mbar_wait_limit(uint64_t* bar, uint32_t phase, int* err, uint64_t limit_ns) {
  if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = global_ns();
  for (int i = 0; i < (1 << 24); ++i) {
    if (mbar_try_wait(bar, phase)) return true;
    if ((i & 255) == 255 && global_ns() - t0 > limit_ns) break;
  }
  set_error(err, QD_DEVERR_TIMEOUT);
  return false;
}

// Add with acquire-release semantics at GPU scope: one round trip that publishes
// this thread's earlier writes (and, after a CTA barrier, the CTA's) and makes the
// writes published before the other arrivals visible to it.
QD_DEV int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// The kernels' wait: about one second.
QD_DEV bool mbar_wait_bounded(uint64_t* bar, uint32_t phase, int* err) {
  return mbar_wait_limit(bar, phase, err, 1000000000ull);
}

// 2D tiled TMA load of the box at (x, y) of a tensor map into shared memory,
// completing on `bar`; x times the element size must be a multiple of 16 bytes.
QD_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before its
// later async-proxy (TMA) ones.
QD_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Global -> shared bulk copy with an L2 cache policy (same alignment rules).
QD_DEV void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// Fetch [src, src + bytes) into L2 with a cache policy; fire and forget.
// src 16-byte aligned, bytes a multiple of 16.
QD_DEV void l2_prefetch_hint(const void* src, uint32_t bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src), "r"(bytes), "l"(pol)
               : "memory");
}

// Global -> shared bulk copy; dst, src 16-byte aligned, bytes a multiple of 16.
QD_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Issue this CTA's share of an L2 prefetch plan from the 32 lanes of one warp.
// The spans are cut into 16 KB pieces dealt round-robin over (CTA, lane), piece
// k of every span before piece k + 1 of any, so the leading bytes of each span
// arrive first. cp.async.bulk.prefetch.L2 is fire-and-forget: no barrier, no
// completion, and a piece never extends past its span.
QD_DEV void l2_prefetch_spans(const L2Prefetch& pf, unsigned cta, unsigned n_cta, int lane) {
  if (pf.base == nullptr || pf.n_spans <= 0 || pf.head_bytes < 16) return;
  constexpr unsigned long long kPiece = 16384;
  const unsigned long long span_max = (unsigned long long)(pf.rows_base + (pf.rows_extra > 0)) * pf.row_bytes;
  const unsigned long long per = (min(pf.head_bytes, span_max) + kPiece - 1) / kPiece;
  const unsigned long long n = per * (unsigned long long)pf.n_spans;
  for (unsigned long long i = cta + (unsigned long long)lane * n_cta; i < n; i += 32ull * n_cta) {
    const int span = (int)(i % (unsigned long long)pf.n_spans);
    const unsigned long long off = (i / (unsigned long long)pf.n_spans) * kPiece;
    const int nr = pf.rows_base + (span < pf.rows_extra ? 1 : 0);
    const unsigned long long bytes = min(pf.head_bytes, (unsigned long long)nr * pf.row_bytes) & ~15ull;
    if (off >= bytes) continue;
    const unsigned long long r0 = (unsigned long long)span * pf.rows_base + (unsigned long long)min(span, pf.rows_extra);
    const unsigned char* src = (const unsigned char*)pf.base + r0 * pf.row_bytes + off;
    const uint32_t sz = (uint32_t)min(kPiece, bytes - off);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(sz) : "memory");
  }
}

}  // namespace qd
