// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/sv.h"

namespace sv {

// Bounded device waits give up after this long (a healthy wait takes
// microseconds).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Every workspace starts with a 256-byte header; the error word is at 0.
constexpr size_t kWorkspaceHeader = 256;

constexpr int kMaxNodes = 128;   // ancestor bitmask width / acceptance walk
constexpr int kMaxSplits = 64;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor-map encoding through the driver entry point (resolved at first use,
// so the library loads on machines without a GPU driver).
CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank, void* base,
                      const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                      CUtensorMapSwizzle swizzle, CUtensorMapL2promotion l2);

// Number of SMs of the current device (cached per device); -1 on failure.
int device_sm_count();

// The 256-row attention kernel (tree_attention_wide.cu): one CTA per (KV
// split, KV head x 256-row group, sequence).  With splits > 1 it writes
// partials (bf16 O / l at part_o, log2-sum-exp at part_lse, [splits][T * Hq])
// for the combine kernel; err is the workspace's error word.
struct WideLaunch {
  int splits;
  void* part_o;
  float* part_lse;
  int* err;
  unsigned long long* trace;
  long long trace_ctas;
};
sv_status launch_wide_attention(const sv_attn_params* p, const WideLaunch& w, cudaStream_t stream);

// The evenly dealt 256-row kernel (tree_attention_dealt.cu): `ctas` resident
// CTAs share the call's weighted (unit, tile) list in equal ranges; pieces of
// units cut by a range boundary go to part_o / part_lse ([ctas][2][256 rows])
// and the last piece of a unit to finish merges them; counters ([units][2],
// zero between calls) count the finished pieces.
struct DealtLaunch {
  int ctas;
  void* part_o;
  float* part_lse;
  int* counters;
  int* err;
  unsigned long long* trace;
  long long trace_ctas;
};
size_t dealt_workspace_bytes(int ctas, int head_dim, long long units);
sv_status launch_dealt_attention(const sv_attn_params* p, const DealtLaunch& w, cudaStream_t stream);

}  // namespace sv
