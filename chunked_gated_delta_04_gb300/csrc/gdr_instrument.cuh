// gdr_instrument.cuh -- the two opt-in instrumentation builds of the kernels, kept out of
// the default build entirely (every macro below expands to nothing unless its flag is set).
//
//  -DGDR_TRACE        phase traces: clock64() cycles between marks of one traced CTA, per-CTA
//                     start/end times (read back through the gdr_debug_trace_* exports).
//  -DGDR_DEBUG_DELAY  delay injection (libgdr_delay.so, `python -m
//                     chunked_gated_delta_04_gb300.build --delay`): GDR_DELAY(site) makes one
//                     role (a copy thread, one warp of an epilogue, a flag publisher, one CTA
//                     of a cluster pair) sleep a short, bounded, pseudo-random time at a
//                     hand-off point, so that it runs late against the roles it hands work
//                     to.  Only timing changes: every result must stay bit for bit the same,
//                     which the tests check against the normal build.
#pragma once

#include <stdint.h>

namespace gdr {
namespace tcx {

#ifdef GDR_DEBUG_DELAY
// Sleeps 0 (one call in four) or 0.25 to 4.3 us, chosen from the CTA, the site and the clock.
__device__ __forceinline__ void debug_delay(uint32_t site) {
  uint32_t x = (blockIdx.x * 0x9E3779B1u) ^ (site * 0x85EBCA77u) ^ (uint32_t)clock64();
  x ^= x >> 15;
  x *= 0x2C1B3C6Du;
  x ^= x >> 12;
  if ((x & 3u) != 0u) __nanosleep(256u + (x >> 20) % 4096u);
}
#define GDR_DELAY(site) gdr::tcx::debug_delay(site)
#else
#define GDR_DELAY(site) \
  do {                  \
  } while (0)
#endif

// Opt-in phase trace (-DGDR_TRACE): thread 0 of CTA GDR_TRACE_BLOCK (default 0) adds the
// clock64() cycles spent between consecutive marks into a per-translation-unit table
// [kernel][mark]; GDR_TRACE_COUNT adds 1 to a slot (e.g. items processed).
#ifdef GDR_TRACE
#ifndef GDR_TRACE_BLOCK
#define GDR_TRACE_BLOCK 0
#endif
static __device__ unsigned long long g_gdr_trace[8][32];
static __device__ unsigned long long g_gdr_cta_span[1024][3];  // per CTA: start, end (ns), SM id
// per CTA, free-form timeline slots (globaltimer ns or counts), written by GDR_TRACE_INFO
static __device__ unsigned long long g_gdr_cta_info[1024][8];
#define GDR_TRACE_NOW()                                              \
  ([]() {                                                            \
    unsigned long long t_;                                           \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));          \
    return t_;                                                       \
  }())
#define GDR_TRACE_INFO_SET(slot, v)                                  \
  do {                                                               \
    if (blockIdx.x < 1024) g_gdr_cta_info[blockIdx.x][slot] = (v);   \
  } while (0)
#define GDR_TRACE_INFO_ADD(slot, v)                                  \
  do {                                                               \
    if (blockIdx.x < 1024) atomicAdd(&g_gdr_cta_info[blockIdx.x][slot], (unsigned long long)(v)); \
  } while (0)
#define GDR_TRACE_CTA_BEGIN()                                                                      \
  do {                                                                                             \
    if (threadIdx.x == 0 && blockIdx.x < 1024) {                                                   \
      unsigned long long t_;                                                                       \
      unsigned int sm_;                                                                            \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                      \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));                                             \
      g_gdr_cta_span[blockIdx.x][0] = t_;                                                          \
      g_gdr_cta_span[blockIdx.x][2] = sm_;                                                         \
    }                                                                                              \
  } while (0)
#define GDR_TRACE_CTA_END()                                                                        \
  do {                                                                                             \
    if (threadIdx.x == 0 && blockIdx.x < 1024) {                                                   \
      unsigned long long t_;                                                                       \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                      \
      g_gdr_cta_span[blockIdx.x][1] = t_;                                                          \
    }                                                                                              \
  } while (0)
#define GDR_TRACE_INIT() unsigned long long gdr_tprev_ = clock64()
#define GDR_TRACE_MARK(kid, slot)                                                                  \
  do {                                                                                             \
    if (threadIdx.x == 0 && blockIdx.x == GDR_TRACE_BLOCK && blockIdx.y == 0 && blockIdx.z == 0) { \
      const unsigned long long now_ = clock64();                                                   \
      atomicAdd(&g_gdr_trace[kid][slot], now_ - gdr_tprev_); /* a reduction: nothing waits on it */ \
      gdr_tprev_ = now_;                                                                           \
    }                                                                                              \
  } while (0)
#define GDR_TRACE_COUNT(kid, slot)                                                                 \
  do {                                                                                             \
    if (threadIdx.x == 0 && blockIdx.x == GDR_TRACE_BLOCK && blockIdx.y == 0 && blockIdx.z == 0)   \
      atomicAdd(&g_gdr_trace[kid][slot], 1ull);                                                    \
  } while (0)
// cycles one thread spends in a region (any thread of the traced CTA)
#define GDR_TRACE_CLK(var) const unsigned long long var = clock64()
#define GDR_TRACE_SINCE(kid, slot, var)                                                            \
  do {                                                                                             \
    if (blockIdx.x == GDR_TRACE_BLOCK) atomicAdd(&g_gdr_trace[kid][slot], clock64() - (var));     \
  } while (0)
#else
#define GDR_TRACE_NOW() 0ull
#define GDR_TRACE_INFO_SET(slot, v) \
  do {                              \
  } while (0)
#define GDR_TRACE_INFO_ADD(slot, v) \
  do {                              \
  } while (0)
#define GDR_TRACE_CTA_BEGIN() \
  do {                        \
  } while (0)
#define GDR_TRACE_CTA_END() \
  do {                      \
  } while (0)
#define GDR_TRACE_INIT() \
  do {                   \
  } while (0)
#define GDR_TRACE_MARK(kid, slot) \
  do {                            \
  } while (0)
#define GDR_TRACE_COUNT(kid, slot) \
  do {                             \
  } while (0)
#define GDR_TRACE_CLK(var) \
  do {                     \
  } while (0)
#define GDR_TRACE_SINCE(kid, slot, var) \
  do {                                  \
  } while (0)
#endif

}  // namespace tcx
}  // namespace gdr
