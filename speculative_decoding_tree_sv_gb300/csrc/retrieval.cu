// SpecPV block retrieval for sm_103a.
//
// SpecPV section 3.2 "Partial Verification": the partial KV cache keeps the
// initial sink blocks, query-dependent retrieved blocks and a local window
// (with the buffer of partially verified tokens at its end), attended as one
// segment; every block's keys are summarised by their element-wise maximum
// and minimum, cached, and scored against the candidate tokens' query states;
// the per-query scores are reduced to one importance per block (max, mean or
// last; Appendix C: mean works best).  Blocks are 16-token pages (Appendix D).
//
// Score of a block for one query q: the largest q . k over keys between the
// block's minimum and maximum, sum_d max(q_d kmax_d, q_d kmin_d)
// = q+ . kmax + q- . kmin with q+ = max(q, 0), q- = min(q, 0).  That form is
// linear in (q+, q-), so the mean over queries (and the mean over heads of the
// last node) is the dot product of the averaged (q+, q-) with the summary: a
// GEMV over the summaries, bound by reading them.  The max reduction needs
// every query's score and runs one query row at a time.
//
// Kernels: page_summary_kernel (one warp per (page, KV head): max/min of the
// page's valid keys, bf16), query_aggregate_kernel (averaged q+, q- per
// (sequence, KV head)), page_score_kernel (one warp per page, the
// sequence's averaged queries staged in shared memory),
// select_kernel (one CTA per sequence: radix select of the k-th largest
// importance, ties to the lower page, then the sink, retrieved and window
// pages written in ascending order).
#include <math.h>

#include <algorithm>

#include "sv_device.cuh"

namespace sv {
namespace retr {

constexpr int kPage = 16;
constexpr int kMaxSortPages = 16384;  // pages per sequence the selection holds in shared memory
constexpr int kSelThreads = 1024;
constexpr int kWarpsPerCta = 8;

// Sink pages, first window page and page count of a context (the same
// regions for every kernel).  Contexts longer than max_ctx_pages pages (a
// host value that should bound them) are cut to that many pages.
struct Regions {
  int n_pages, sink, first_window;
};

__device__ __forceinline__ int clamp_len(int L, int max_ctx_pages) { return min(L, max_ctx_pages * kPage); }

__device__ __forceinline__ Regions regions(int L, int sink_tokens, int window_tokens) {
  Regions r;
  r.n_pages = (L + kPage - 1) / kPage;
  r.sink = min(r.n_pages, (sink_tokens + kPage - 1) / kPage);
  r.first_window = max(r.sink, min(r.n_pages, max(0, L - window_tokens) / kPage));
  return r;
}

__device__ __forceinline__ int list_length(int L, int sink_tokens, int window_tokens, int topk) {
  const Regions r = regions(L, sink_tokens, window_tokens);
  return r.sink + min(topk, r.first_window - r.sink) + (r.n_pages - r.first_window);
}

// ------------------------------------------------------------------ summaries

struct SumParams {
  const __nv_bfloat16* k_cache;  // [num_pages, Hkv, 16, D]
  __nv_bfloat16* summ;           // [num_pages, Hkv, 2, D]: max, then min
  const int* block_table;
  const int* ctx_lens;
  const int* first_page;  // optional [B]
  int* err;
  int num_pages;
  int num_kv_heads;
  int max_pages_per_seq;
};

template <int D>
__global__ void __launch_bounds__(256) page_summary_kernel(const __grid_constant__ SumParams p) {
  constexpr int E = D / 32;  // elements per lane
  const int b = blockIdx.y;
  const int w = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int L = p.ctx_lens[b];
  const int n_pages = (L + kPage - 1) / kPage;
  const int lp = (p.first_page != nullptr ? max(0, p.first_page[b]) : 0) + w / p.num_kv_heads;
  const int h = w % p.num_kv_heads;
  if (lp >= n_pages) return;
  if (lp >= p.max_pages_per_seq) {
    if (lane == 0) report_error(p.err, SV_DEVERR_BAD_PAGE);
    return;
  }
  const int phys = p.block_table[static_cast<size_t>(b) * p.max_pages_per_seq + lp];
  if (phys < 0 || phys >= p.num_pages) {
    if (lane == 0) report_error(p.err, SV_DEVERR_BAD_PAGE);
    return;
  }
  const int valid = min(kPage, L - lp * kPage);
  const __nv_bfloat16* src = p.k_cache + (static_cast<size_t>(phys) * p.num_kv_heads + h) * kPage * D + lane * E;
  float mx[E], mn[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    mx[e] = -INFINITY;
    mn[e] = INFINITY;
  }
  // all sixteen rows are requested before any is used (rows past the valid
  // tokens repeat row 0, which cannot change a max or a min)
  uint32_t rows[kPage][E / 2];
#pragma unroll
  for (int t = 0; t < kPage; ++t) {
    const int tt = t < valid ? t : 0;
    if constexpr (E == 4) {
      const uint2 x = __ldg(reinterpret_cast<const uint2*>(src + tt * D));
      rows[t][0] = x.x;
      rows[t][1] = x.y;
    } else {
      rows[t][0] = __ldg(reinterpret_cast<const unsigned int*>(src + tt * D));
    }
  }
#pragma unroll
  for (int t = 0; t < kPage; ++t) {
    const uint32_t* v = rows[t];
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {
      const float lo = __uint_as_float(v[e] << 16), hi = __uint_as_float(v[e] & 0xFFFF0000u);
      mx[2 * e] = fmaxf(mx[2 * e], lo);
      mn[2 * e] = fminf(mn[2 * e], lo);
      mx[2 * e + 1] = fmaxf(mx[2 * e + 1], hi);
      mn[2 * e + 1] = fminf(mn[2 * e + 1], hi);
    }
  }
  // max and min of bf16 values are bf16 values: the conversion back is exact
  __nv_bfloat16* dst = p.summ + (static_cast<size_t>(phys) * p.num_kv_heads + h) * 2 * D + lane * E;
  uint32_t omx[E / 2], omn[E / 2];
#pragma unroll
  for (int e = 0; e < E / 2; ++e) {
    omx[e] = pack_bf16x2(mx[2 * e], mx[2 * e + 1]);
    omn[e] = pack_bf16x2(mn[2 * e], mn[2 * e + 1]);
  }
  if constexpr (E == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(omx[0], omx[1]);
    *reinterpret_cast<uint2*>(dst + D) = make_uint2(omn[0], omn[1]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = omx[0];
    *reinterpret_cast<uint32_t*>(dst + D) = omn[0];
  }
}

// ------------------------------------------------------------------ queries

struct AggParams {
  const __nv_bfloat16* q;  // [T, Hq, D]
  const int* cu_nodes;
  float* qa;               // [B, Hkv, 2, D]: averaged q+ and q-
  int num_q_heads;
  int group;
  int last_only;
};

// The mean over the used queries of q+ and q-, split by KV head: the sum
// over KV heads of qa . (kmax, kmin) is then the mean score.  One CTA per
// (KV head, sequence), 1024 threads: a thread owns eight dimensions of every
// (1024 / (D / 8))-th query row and requests all its rows with 16-byte loads
// before summing them, so the whole group arrives in one round trip; the
// row slices are then folded within each warp by shuffles and across warps
// in shared memory (a fixed order: the result does not depend on timing).
template <int D>
__global__ void __launch_bounds__(1024) query_aggregate_kernel(const __grid_constant__ AggParams p) {
  constexpr int kChunks = D / 8;             // 16-byte chunks of a row
  constexpr int kSlices = 1024 / kChunks;    // row slices
  constexpr int kWarpSlices = 32 / kChunks;  // slices inside one warp
  __shared__ float red[2][32][D];
  const int kvh = blockIdx.x;
  const int b = blockIdx.y;
  const int c = threadIdx.x % kChunks;
  const int slice = threadIdx.x / kChunks;
  const int n0 = p.cu_nodes[b];
  const int N = p.cu_nodes[b + 1] - n0;
  const int i0 = p.last_only ? max(0, N - 1) : 0;
  const int used = N - i0;
  const int rows = used * p.group;
  float pos[8], neg[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) pos[e] = neg[e] = 0.f;
#pragma unroll 8
  for (int r = slice; r < rows; r += kSlices) {
    const int i = i0 + r / p.group, g = r % p.group;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(
        p.q + (static_cast<size_t>(n0 + i) * p.num_q_heads + kvh * p.group + g) * D + c * 8));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
      pos[2 * e] += fmaxf(lo, 0.f);
      neg[2 * e] += fminf(lo, 0.f);
      pos[2 * e + 1] += fmaxf(hi, 0.f);
      neg[2 * e + 1] += fminf(hi, 0.f);
    }
  }
  // slices of one warp: lanes c, c + kChunks, ... hold the same dimensions
#pragma unroll
  for (int o = kChunks; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      pos[e] += __shfl_xor_sync(0xffffffffu, pos[e], o);
      neg[e] += __shfl_xor_sync(0xffffffffu, neg[e], o);
    }
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) < kChunks) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      red[0][warp][c * 8 + e] = pos[e];
      red[1][warp][c * 8 + e] = neg[e];
    }
  }
  __syncthreads();
  static_assert(kWarpSlices >= 1 && 2 * D <= 1024, "row slices");
  if (threadIdx.x < 2 * D) {
    const int half = threadIdx.x / D, d = threadIdx.x % D;
    float acc = 0.f;
    for (int w = 0; w < 32; ++w) acc += red[half][w][d];
    const float scale = used > 0 ? 1.f / (static_cast<float>(used) * p.num_q_heads) : 0.f;
    p.qa[(static_cast<size_t>(b) * gridDim.x + kvh) * 2 * D + half * D + d] = acc * scale;
  }
}

// ------------------------------------------------------------------ scores

struct ScoreParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* summ;
  const float* qa;
  const int* block_table;
  const int* ctx_lens;
  const int* cu_nodes;
  float* scores;  // [B, max_ctx_pages]; -inf for pages that are not candidates
  int* err;
  int num_pages;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int max_pages_per_seq;
  int max_ctx_pages;
  int sink_tokens;
  int window_tokens;
  int reduce_max;
};

template <int D>
__global__ void __launch_bounds__(256) page_score_kernel(const __grid_constant__ ScoreParams p) {
  constexpr int E = D / 32;
  extern __shared__ float qa_s[];  // mean / last: this sequence's qa, [Hkv][2][D]
  const int b = blockIdx.y;
  const int lp = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (!p.reduce_max) {
    // every warp of the CTA scores a page of this sequence against the same
    // averaged queries: read them once per CTA
    const float4* src = reinterpret_cast<const float4*>(p.qa + static_cast<size_t>(b) * p.num_kv_heads * 2 * D);
    float4* dst = reinterpret_cast<float4*>(qa_s);
    for (int i = threadIdx.x; i < p.num_kv_heads * 2 * D / 4; i += blockDim.x) dst[i] = src[i];
    __syncthreads();
  }
  if (lp >= p.max_ctx_pages) return;
  const int L = clamp_len(p.ctx_lens[b], p.max_ctx_pages);
  const Regions rg = regions(L, p.sink_tokens, p.window_tokens);
  float out = -INFINITY;
  if (lp >= rg.sink && lp < rg.first_window && lp < p.max_pages_per_seq) {
    int phys = p.block_table[static_cast<size_t>(b) * p.max_pages_per_seq + lp];
    if (phys < 0 || phys >= p.num_pages) {
      if (lane == 0) report_error(p.err, SV_DEVERR_BAD_PAGE);
      phys = 0;
    }
    if (!p.reduce_max) {
      float acc = 0.f;
#pragma unroll 8
      for (int kvh = 0; kvh < p.num_kv_heads; ++kvh) {
        // this lane's E maxima and E minima (bf16, one 4- or 8-byte load each)
        const __nv_bfloat16* s = p.summ + (static_cast<size_t>(phys) * p.num_kv_heads + kvh) * 2 * D + lane * E;
        uint32_t mx[E / 2], mn[E / 2];
        if constexpr (E == 4) {
          const uint2 a2 = __ldg(reinterpret_cast<const uint2*>(s));
          const uint2 b2 = __ldg(reinterpret_cast<const uint2*>(s + D));
          mx[0] = a2.x;
          mx[1] = a2.y;
          mn[0] = b2.x;
          mn[1] = b2.y;
        } else {
          mx[0] = __ldg(reinterpret_cast<const unsigned int*>(s));
          mn[0] = __ldg(reinterpret_cast<const unsigned int*>(s + D));
        }
        const float* a = qa_s + kvh * 2 * D + lane * E;
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
          acc += a[2 * e] * __uint_as_float(mx[e] << 16) + a[2 * e + 1] * __uint_as_float(mx[e] & 0xFFFF0000u);
          acc += a[D + 2 * e] * __uint_as_float(mn[e] << 16) +
                 a[D + 2 * e + 1] * __uint_as_float(mn[e] & 0xFFFF0000u);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      out = acc;
    } else {
      const int n0 = p.cu_nodes[b];
      const int rows = (p.cu_nodes[b + 1] - n0) * p.group;
      float best = -INFINITY;
      for (int kvh = 0; kvh < p.num_kv_heads; ++kvh) {
        const __nv_bfloat16* s = p.summ + (static_cast<size_t>(phys) * p.num_kv_heads + kvh) * 2 * D + lane * E;
        float kmx[E], kmn[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          kmx[e] = __bfloat162float(s[e]);
          kmn[e] = __bfloat162float(s[D + e]);
        }
        for (int r0 = 0; r0 < rows; r0 += 4) {
          float part[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            part[u] = 0.f;
            const int r = min(r0 + u, rows - 1);
            const __nv_bfloat16* qr =
                p.q + (static_cast<size_t>(n0 + r / p.group) * p.num_q_heads + kvh * p.group + r % p.group) * D +
                lane * E;
#pragma unroll
            for (int e = 0; e < E; ++e) {
              const float v = __bfloat162float(qr[e]);
              part[u] += fmaxf(v * kmx[e], v * kmn[e]);
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int u = 0; u < 4; ++u) part[u] += __shfl_xor_sync(0xffffffffu, part[u], o);
#pragma unroll
          for (int u = 0; u < 4; ++u) best = fmaxf(best, part[u]);  // repeats of the last row are harmless
        }
      }
      out = best;
    }
  }
  if (lane == 0) p.scores[static_cast<size_t>(b) * p.max_ctx_pages + lp] = out;
}

// ------------------------------------------------------------------ selection

struct SelParams {
  const float* scores;
  const int* ctx_lens;
  int* kv_pages;
  int* cu_kv_pages;
  int* err;
  int batch;
  int max_ctx_pages;
  int sink_tokens;
  int window_tokens;
  int topk;
};

// Order-preserving map of a float to an unsigned integer.
__device__ __forceinline__ uint32_t ordered(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive prefix sum of one int per thread (kSelThreads).
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  const int before = (warp > 0 ? scratch[warp - 1] : 0) + x - v;
  if (total != nullptr) *total = scratch[kSelThreads / 32 - 1];
  __syncthreads();
  return before;
}

// One CTA per sequence.  The topk largest importances among the candidate
// pages are found by a radix select on their order-preserving 32-bit codes
// (four passes of eight bits): it yields the k-th largest code T and how
// many pages with code T still belong to the top k, which are then the
// lowest such pages.  Sink, retrieved and window pages are marked in a
// bitmap and written in ascending order.
__global__ void __launch_bounds__(kSelThreads) select_kernel(const __grid_constant__ SelParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint32_t* code = reinterpret_cast<uint32_t*>(smem_raw);           // [kMaxSortPages]
  uint32_t* bits = code + kMaxSortPages;                             // [kMaxSortPages / 32]
  int* hist = reinterpret_cast<int*>(bits + kMaxSortPages / 32);     // [256]
  int* scratch = hist + 256;                                         // [32 + 4]
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid == 0 && p.ctx_lens[b] > p.max_ctx_pages * kPage) report_error(p.err, SV_DEVERR_BAD_PAGE);
  const int L = clamp_len(p.ctx_lens[b], p.max_ctx_pages);
  const Regions rg = regions(L, p.sink_tokens, p.window_tokens);
  const int ncand = rg.first_window - rg.sink;
  const int k = min(p.topk, ncand);
  // where this sequence's list starts: the lengths of the earlier lists
  int part = 0;
  for (int j = tid; j < b; j += kSelThreads)
    part += list_length(clamp_len(p.ctx_lens[j], p.max_ctx_pages), p.sink_tokens, p.window_tokens, p.topk);
  int offset = 0;
  block_exclusive_scan(part, scratch, &offset);
  for (int i = tid; i < ncand; i += kSelThreads)
    code[i] = ordered(p.scores[static_cast<size_t>(b) * p.max_ctx_pages + rg.sink + i]);
  for (int i = tid; i < kMaxSortPages / 32; i += kSelThreads) bits[i] = 0u;
  // radix select of the k-th largest code
  uint32_t prefix = 0u, mask = 0u;
  int remaining = k;
  volatile int* sel = scratch + 32;  // chosen digit, count above it
  for (int shift = 24; shift >= 0 && k > 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    // Scores of one sequence share their high bits, so most codes fall into
    // a few bins: lanes holding the same digit add once, as a group.
    for (int base = 0; base < ncand; base += kSelThreads) {
      const int i = base + tid;
      const uint32_t c = i < ncand ? code[i] : 0u;
      const bool part = i < ncand && (c & mask) == prefix;
      const uint32_t key = part ? (c >> shift) & 255u : 0xFFFFFFFFu;
      const uint32_t peers = __match_any_sync(0xffffffffu, key);
      if (part && (tid & 31) == __ffs(peers) - 1) atomicAdd(&hist[key], __popc(peers));
    }
    __syncthreads();
    if (tid < 32) {
      // lane l holds digits 255 - 8l .. 248 - 8l (high digits first)
      int cnt[8], sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        cnt[e] = hist[255 - 8 * tid - e];
        sum += cnt[e];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      int above = incl - sum;  // codes in higher digits than this lane's
      const bool here = above < remaining && above + sum >= remaining;
      if (here) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (above + cnt[e] >= remaining) {
            sel[0] = 255 - 8 * tid - e;
            sel[1] = above;
            break;
          }
          above += cnt[e];
        }
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sel[0]) << shift;
    mask |= 255u << shift;
    remaining -= sel[1];
    __syncthreads();
  }
  // codes above the threshold are retrieved; of those equal to it, the
  // `remaining` lowest pages (candidates are stored in page order)
  const int per = (ncand + kSelThreads - 1) / kSelThreads;
  const int c0 = min(ncand, tid * per), c1 = min(ncand, c0 + per);
  int eq = 0;
  if (k > 0)
    for (int i = c0; i < c1; ++i) eq += (code[i] == prefix) ? 1 : 0;
  int eq_before = block_exclusive_scan(eq, scratch, nullptr);
  if (k > 0) {
    for (int i = c0; i < c1; ++i) {
      const uint32_t c = code[i];
      bool take = c > prefix;
      if (c == prefix) take = eq_before++ < remaining;
      if (take) {
        const int page = rg.sink + i;
        atomicOr(&bits[page >> 5], 1u << (page & 31));
      }
    }
  }
  for (int page = tid; page < rg.n_pages; page += kSelThreads)
    if (page < rg.sink || page >= rg.first_window) atomicOr(&bits[page >> 5], 1u << (page & 31));
  __syncthreads();
  const int words = (rg.n_pages + 31) / 32;
  const int wper = (words + kSelThreads - 1) / kSelThreads;  // words per thread
  const int w0 = min(words, tid * wper), w1 = min(words, w0 + wper);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(bits[w]);
  int pos = offset + block_exclusive_scan(cnt, scratch, nullptr);
  for (int w = w0; w < w1; ++w) {
    uint32_t m = bits[w];
    while (m) {
      const int bit = __ffs(m) - 1;
      m &= m - 1;
      p.kv_pages[pos++] = w * 32 + bit;
    }
  }
  if (tid == 0) {
    p.cu_kv_pages[b + 1] = offset + list_length(L, p.sink_tokens, p.window_tokens, p.topk);
    if (b == 0) p.cu_kv_pages[0] = 0;
  }
}

constexpr size_t kSelSmemBytes = kMaxSortPages * 4 + kMaxSortPages / 8 + 256 * 4 + 36 * 4;

// ------------------------------------------------------------------ list extension

struct ExtendParams {
  const int* ref_pages;  // the lists made at the last refresh
  const int* ref_cu;
  const int* ref_ctx_lens;
  const int* ctx_lens;
  int* kv_pages;
  int* cu_kv_pages;
  int* err;
};

// The partial cache between refreshes: the refresh's list plus every page
// the buffer of partially verified tokens has grown into since (SpecPV
// section 3.3).  One CTA per sequence; the start of its list is the sum of
// the earlier sequences' lengths.
__device__ __forceinline__ int extended_length(const ExtendParams& p, int j) {
  const int n_ref = p.ref_cu[j + 1] - p.ref_cu[j];
  const int ref_pages = (p.ref_ctx_lens[j] + kPage - 1) / kPage;
  const int now_pages = (p.ctx_lens[j] + kPage - 1) / kPage;
  return n_ref + max(0, now_pages - max(ref_pages, 0));
}

__global__ void __launch_bounds__(256) list_extend_kernel(const __grid_constant__ ExtendParams p) {
  __shared__ int red[256];
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  int part = 0;
  for (int j = tid; j < b; j += blockDim.x) part += extended_length(p, j);
  red[tid] = part;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if (tid < s) red[tid] += red[tid + s];
    __syncthreads();
  }
  const int offset = red[0];
  const int r0 = p.ref_cu[b], n_ref = p.ref_cu[b + 1] - r0;
  const int ref_pages = (p.ref_ctx_lens[b] + kPage - 1) / kPage;
  const int now_pages = (p.ctx_lens[b] + kPage - 1) / kPage;
  if (tid == 0 && p.ctx_lens[b] < p.ref_ctx_lens[b]) report_error(p.err, SV_DEVERR_BAD_PAGE);
  for (int i = tid; i < n_ref; i += blockDim.x) p.kv_pages[offset + i] = p.ref_pages[r0 + i];
  for (int i = tid; i < now_pages - ref_pages; i += blockDim.x) p.kv_pages[offset + n_ref + i] = ref_pages + i;
  if (tid == 0) {
    p.cu_kv_pages[b + 1] = offset + n_ref + max(0, now_pages - ref_pages);
    if (b == 0) p.cu_kv_pages[0] = 0;
  }
}

// SpecPV section 3.3: before a full verification the partially verified
// tokens are prepended to the new candidates.  One CTA per sequence b writes
// its combined tree at the offset sum over earlier sequences of (buffered +
// candidate nodes): the buffered tokens as a chain from the root (node j,
// parent j - 1), then the candidate tree with ids shifted by the buffer's
// length, its root's parent being the last buffered token.
struct FullTreeParams {
  const int* cand_parents;
  const int* cand_tokens;
  const int* cand_cu;
  const int* buffer_tokens;
  const int* buffer_cu;
  int* parents;
  int* tokens;
  int* cu_nodes;
  int* err;
};

__device__ __forceinline__ int combined_nodes(const FullTreeParams& p, int b) {
  return max(0, p.buffer_cu[b + 1] - p.buffer_cu[b]) + max(0, p.cand_cu[b + 1] - p.cand_cu[b]);
}

__global__ void __launch_bounds__(256) full_tree_kernel(const __grid_constant__ FullTreeParams p) {
  __shared__ int red[256];
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  int part = 0;
  for (int j = tid; j < b; j += blockDim.x) part += combined_nodes(p, j);
  red[tid] = part;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if (tid < s) red[tid] += red[tid + s];
    __syncthreads();
  }
  const int offset = red[0];
  const int b0 = p.buffer_cu[b], nb = p.buffer_cu[b + 1] - b0;
  const int c0 = p.cand_cu[b], n = p.cand_cu[b + 1] - c0;
  if (tid == 0 && (nb < 0 || n < 1 || max(0, nb) + n > kMaxNodes)) report_error(p.err, SV_DEVERR_BAD_TREE);
  const int nbv = max(0, nb), nv = max(0, n);
  for (int j = tid; j < nbv; j += blockDim.x) {
    p.parents[offset + j] = j - 1;
    p.tokens[offset + j] = p.buffer_tokens[b0 + j];
  }
  for (int i = tid; i < nv; i += blockDim.x) {
    int par = nbv - 1;  // the candidate root hangs below the chain (-1: no buffer)
    if (i > 0) {
      const int cp = p.cand_parents[c0 + i];
      if (cp < 0 || cp >= i) report_error(p.err, SV_DEVERR_BAD_PARENT);
      par = nbv + cp;
    }
    p.parents[offset + nbv + i] = par;
    p.tokens[offset + nbv + i] = p.cand_tokens[c0 + i];
  }
  if (tid == 0) {
    p.cu_nodes[b + 1] = offset + nbv + nv;
    if (b == 0) p.cu_nodes[0] = 0;
  }
}

}  // namespace retr
}  // namespace sv

extern "C" {

sv_status sv_partial_list_extend(const int* ref_pages, const int* ref_cu, const int* ref_ctx_lens,
                                 const int* ctx_lens, int batch, int* kv_pages, int* cu_kv_pages,
                                 void* workspace, size_t workspace_bytes, sv_stream_t stream) {
  using namespace sv;
  if (!ref_pages || !ref_cu || !ref_ctx_lens || !ctx_lens || !kv_pages || !cu_kv_pages || batch < 1)
    return SV_ERR_INVALID_ARG;
  if (workspace != nullptr && workspace_bytes < kWorkspaceHeader) return SV_ERR_WORKSPACE;
  retr::ExtendParams p;
  p.ref_pages = ref_pages;
  p.ref_cu = ref_cu;
  p.ref_ctx_lens = ref_ctx_lens;
  p.ctx_lens = ctx_lens;
  p.kv_pages = kv_pages;
  p.cu_kv_pages = cu_kv_pages;
  p.err = static_cast<int*>(workspace);
  retr::list_extend_kernel<<<batch, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_specpv_full_trees(const int* cand_parents, const int* cand_tokens, const int* cand_cu,
                               const int* buffer_tokens, const int* buffer_cu, int batch, int* parents,
                               int* tokens, int* cu_nodes, void* workspace, size_t workspace_bytes,
                               sv_stream_t stream) {
  using namespace sv;
  if (!cand_parents || !cand_tokens || !cand_cu || !buffer_cu || !parents || !tokens || !cu_nodes || batch < 1)
    return SV_ERR_INVALID_ARG;
  if (workspace != nullptr && workspace_bytes < kWorkspaceHeader) return SV_ERR_WORKSPACE;
  if (batch > 65535) return SV_ERR_UNSUPPORTED;
  retr::FullTreeParams p;
  p.cand_parents = cand_parents;
  p.cand_tokens = cand_tokens;
  p.cand_cu = cand_cu;
  p.buffer_tokens = buffer_tokens;
  p.buffer_cu = buffer_cu;
  p.parents = parents;
  p.tokens = tokens;
  p.cu_nodes = cu_nodes;
  p.err = static_cast<int*>(workspace);
  retr::full_tree_kernel<<<batch, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_verify_kind sv_specpv_next(const sv_specpv_seq* seq, int step_tokens, int buffer_limit) {
  if (seq == nullptr || !seq->has_partial_cache) return SV_VERIFY_FULL;
  return seq->buffer_tokens + step_tokens > buffer_limit ? SV_VERIFY_FULL : SV_VERIFY_PARTIAL;
}

sv_status sv_specpv_after(sv_specpv_seq* seq, sv_verify_kind kind, int ctx_len_after) {
  if (seq == nullptr || ctx_len_after < 0) return SV_ERR_INVALID_ARG;
  if (kind == SV_VERIFY_FULL) {
    seq->has_partial_cache = 1;
    seq->refresh_ctx_len = ctx_len_after;
    seq->buffer_tokens = 0;
    return SV_OK;
  }
  if (kind != SV_VERIFY_PARTIAL || !seq->has_partial_cache || ctx_len_after < seq->refresh_ctx_len)
    return SV_ERR_INVALID_ARG;
  seq->buffer_tokens = ctx_len_after - seq->refresh_ctx_len;
  return SV_OK;
}


sv_status sv_kv_page_summaries(const void* k_cache, int num_pages, int num_kv_heads, int head_dim, int page_size,
                               const int* block_table, int max_pages_per_seq, const int* ctx_lens,
                               const int* first_page, int batch, int max_ctx_pages, void* summaries,
                               void* workspace, size_t workspace_bytes, sv_stream_t stream) {
  using namespace sv;
  if (!k_cache || !block_table || !ctx_lens || !summaries) return SV_ERR_INVALID_ARG;
  if (num_pages < 1 || num_kv_heads < 1 || batch < 1 || max_pages_per_seq < 1 || max_ctx_pages < 0)
    return SV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return SV_ERR_UNSUPPORTED;
  if (page_size != retr::kPage) return SV_ERR_UNSUPPORTED;
  if (!aligned16(k_cache) || !aligned16(summaries)) return SV_ERR_INVALID_ARG;
  if (workspace != nullptr && workspace_bytes < kWorkspaceHeader) return SV_ERR_WORKSPACE;
  if (batch > 65535) return SV_ERR_UNSUPPORTED;
  if (max_ctx_pages == 0) return SV_OK;
  retr::SumParams p;
  p.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  p.summ = static_cast<__nv_bfloat16*>(summaries);
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.first_page = first_page;
  p.err = static_cast<int*>(workspace);
  p.num_pages = num_pages;
  p.num_kv_heads = num_kv_heads;
  p.max_pages_per_seq = max_pages_per_seq;
  const long long warps = static_cast<long long>(max_ctx_pages) * num_kv_heads;
  const dim3 grid(static_cast<unsigned>((warps + retr::kWarpsPerCta - 1) / retr::kWarpsPerCta), batch, 1);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (head_dim == 128) retr::page_summary_kernel<128><<<grid, 256, 0, s>>>(p);
  else retr::page_summary_kernel<64><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_retrieve_pages_workspace_size(int batch, int num_kv_heads, int head_dim, int max_ctx_pages,
                                           size_t* bytes) {
  using namespace sv;
  if (bytes == nullptr || batch < 1 || num_kv_heads < 1 || head_dim < 1 || max_ctx_pages < 0)
    return SV_ERR_INVALID_ARG;
  *bytes = kWorkspaceHeader +
           align_up(static_cast<size_t>(batch) * num_kv_heads * 2 * head_dim * sizeof(float), 256) +
           align_up(static_cast<size_t>(batch) * max_ctx_pages * sizeof(float), 256);
  return SV_OK;
}

sv_status sv_retrieve_pages(const sv_retrieve_params* rp, sv_stream_t stream) {
  using namespace sv;
  if (rp == nullptr) return SV_ERR_INVALID_ARG;
  const sv_retrieve_params& r = *rp;
  if (!r.q || !r.summaries || !r.block_table || !r.ctx_lens || !r.cu_nodes || !r.kv_pages || !r.cu_kv_pages)
    return SV_ERR_INVALID_ARG;
  if (r.batch < 1 || r.num_q_heads < 1 || r.num_kv_heads < 1 || r.num_q_heads % r.num_kv_heads != 0 ||
      r.num_pages < 1 || r.max_pages_per_seq < 1 || r.max_ctx_pages < 0 || r.sink_tokens < 0 ||
      r.window_tokens < 0 || r.topk < 0 || r.reduce < SV_REDUCE_MEAN || r.reduce > SV_REDUCE_LAST ||
      r.total_nodes < 1)
    return SV_ERR_INVALID_ARG;
  if (r.head_dim != 64 && r.head_dim != 128) return SV_ERR_UNSUPPORTED;
  if (r.page_size != retr::kPage) return SV_ERR_UNSUPPORTED;
  if (r.max_ctx_pages > retr::kMaxSortPages || r.max_ctx_pages > r.max_pages_per_seq) return SV_ERR_UNSUPPORTED;
  if (static_cast<size_t>(r.num_kv_heads) * 2 * r.head_dim * sizeof(float) > 227 * 1024)
    return SV_ERR_UNSUPPORTED;  // the averaged queries of a sequence must fit in shared memory
  if (!aligned16(r.q) || !aligned16(r.summaries)) return SV_ERR_INVALID_ARG;
  const long long per_seq =
      (r.sink_tokens + retr::kPage - 1) / retr::kPage + static_cast<long long>(r.topk) +
      (r.window_tokens + retr::kPage - 1) / retr::kPage + 1;
  if (r.kv_pages_capacity < static_cast<size_t>(r.batch) * static_cast<size_t>(
                                std::min<long long>(per_seq, r.max_ctx_pages)))
    return SV_ERR_INVALID_ARG;
  size_t need = 0;
  sv_retrieve_pages_workspace_size(r.batch, r.num_kv_heads, r.head_dim, r.max_ctx_pages, &need);
  if (r.workspace == nullptr || r.workspace_bytes < need) return SV_ERR_WORKSPACE;
  if (r.batch > 65535) return SV_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(r.workspace);
  float* qa = reinterpret_cast<float*>(ws + kWorkspaceHeader);
  float* scores = r.scores != nullptr
                      ? r.scores
                      : reinterpret_cast<float*>(
                            ws + kWorkspaceHeader +
                            align_up(static_cast<size_t>(r.batch) * r.num_kv_heads * 2 * r.head_dim * sizeof(float),
                                     256));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int G = r.num_q_heads / r.num_kv_heads;
  const bool use_max = r.reduce == SV_REDUCE_MAX;
  if (!use_max) {
    retr::AggParams a;
    a.q = static_cast<const __nv_bfloat16*>(r.q);
    a.cu_nodes = r.cu_nodes;
    a.qa = qa;
    a.num_q_heads = r.num_q_heads;
    a.group = G;
    a.last_only = r.reduce == SV_REDUCE_LAST ? 1 : 0;
    const dim3 grid(r.num_kv_heads, r.batch, 1);
    if (r.head_dim == 128) retr::query_aggregate_kernel<128><<<grid, 1024, 0, s>>>(a);
    else retr::query_aggregate_kernel<64><<<grid, 1024, 0, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  }
  if (r.max_ctx_pages > 0) {
    retr::ScoreParams sp;
    sp.q = static_cast<const __nv_bfloat16*>(r.q);
    sp.summ = static_cast<const __nv_bfloat16*>(r.summaries);
    sp.qa = qa;
    sp.block_table = r.block_table;
    sp.ctx_lens = r.ctx_lens;
    sp.cu_nodes = r.cu_nodes;
    sp.scores = scores;
    sp.err = reinterpret_cast<int*>(ws);
    sp.num_pages = r.num_pages;
    sp.num_q_heads = r.num_q_heads;
    sp.num_kv_heads = r.num_kv_heads;
    sp.group = G;
    sp.max_pages_per_seq = r.max_pages_per_seq;
    sp.max_ctx_pages = r.max_ctx_pages;
    sp.sink_tokens = r.sink_tokens;
    sp.window_tokens = r.window_tokens;
    sp.reduce_max = use_max ? 1 : 0;
    const dim3 grid((r.max_ctx_pages + retr::kWarpsPerCta - 1) / retr::kWarpsPerCta, r.batch, 1);
    const size_t qa_smem = use_max ? 0 : static_cast<size_t>(r.num_kv_heads) * 2 * r.head_dim * sizeof(float);
    if (qa_smem > 48 * 1024) {
      const cudaError_t e = r.head_dim == 128
                                ? cudaFuncSetAttribute(retr::page_score_kernel<128>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(qa_smem))
                                : cudaFuncSetAttribute(retr::page_score_kernel<64>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(qa_smem));
      if (e != cudaSuccess) return SV_ERR_CUDA;
    }
    if (r.head_dim == 128) retr::page_score_kernel<128><<<grid, 256, qa_smem, s>>>(sp);
    else retr::page_score_kernel<64><<<grid, 256, qa_smem, s>>>(sp);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  }
  retr::SelParams sel;
  sel.scores = scores;
  sel.ctx_lens = r.ctx_lens;
  sel.kv_pages = r.kv_pages;
  sel.cu_kv_pages = r.cu_kv_pages;
  sel.err = reinterpret_cast<int*>(ws);
  sel.batch = r.batch;
  sel.max_ctx_pages = r.max_ctx_pages;
  sel.sink_tokens = r.sink_tokens;
  sel.window_tokens = r.window_tokens;
  sel.topk = r.topk;
  if (cudaFuncSetAttribute(retr::select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(retr::kSelSmemBytes)) != cudaSuccess)
    return SV_ERR_CUDA;
  retr::select_kernel<<<r.batch, retr::kSelThreads, retr::kSelSmemBytes, s>>>(sel);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"
