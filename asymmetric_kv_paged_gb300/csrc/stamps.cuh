// Start-up and epilogue timestamps of the split-KV kernel, for a profiling
// build of the library only.  With AKP_STAMPS defined (build.build(stamps=True),
// a library of its own next to the default one), each CTA below kStampCtas
// writes the %globaltimer value (ns) at fixed points of its run into
// g_stamps[cta][event]; attn_debug_stamps copies the array out.  Without it,
// AKP_STAMP expands to nothing and the kernels are the default build's.
#pragma once

#include <cstdint>

namespace akp {

constexpr int kStampCtas = 160;
constexpr int kStampEvents = 16;

// Event indices (times unless noted).
enum StampEvent : int {
  kStampStart = 0,      // first instruction of thread 0
  kStampHead = 1,       // head record read (segment range known)
  kStampReady = 2,      // barriers initialised and TMEM allocated
  kStampFirstLoad = 3,  // producer: first tile's K/V requested (TMA issue / slots resolved)
  kStampFirstQ = 4,     // converters: first block's Q staged
  kStampFirstQK = 5,    // first Q.K^T issued
  kStampFirstS = 6,     // softmax: first S tile ready
  kStampLastPV = 7,     // last P.V issued
  kStampEpiBegin = 8,   // softmax: last segment's epilogue begins (its P.V done)
  kStampEpiEnd = 9,     // softmax: last segment's epilogue ends
  kStampEnd = 10,       // all roles done (before TMEM is freed)
  kStampSegs = 11,      // value: segments of the CTA
  kStampTiles = 12,     // value: key tiles of the CTA
  kStampLookup = 13,    // producer: first tile's page-table entries read (TMA paths)
  kStampSm = 14,        // value: the SM the CTA runs on (%smid)
};

}  // namespace akp

// The translation unit that stamps defines the array (akp::g_stamps, of
// kStampCtas * kStampEvents values) before its kernels.
#ifdef AKP_STAMPS
#define AKP_STAMP_VALUE(ev, v)                                                    \
  do {                                                                            \
    if (blockIdx.x < (unsigned)::akp::kStampCtas)                                 \
      ::akp::g_stamps[blockIdx.x * ::akp::kStampEvents + (ev)] =                  \
          (unsigned long long)(v);                                                \
  } while (0)
#define AKP_STAMP(ev)                                                             \
  do {                                                                            \
    unsigned long long t_;                                                        \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                       \
    AKP_STAMP_VALUE(ev, t_);                                                      \
  } while (0)
#define AKP_STAMP_SMID(ev)                                                        \
  do {                                                                            \
    unsigned sm_;                                                                 \
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));                             \
    AKP_STAMP_VALUE(ev, sm_);                                                     \
  } while (0)
#else
#define AKP_STAMP_SMID(ev) \
  do {                     \
  } while (0)
#define AKP_STAMP_VALUE(ev, v) \
  do {                         \
  } while (0)
#define AKP_STAMP(ev) \
  do {                \
  } while (0)
#endif
