// Greedy (temperature 0) acceptance of a verified draft tree.
//
// SpecBlock Appendix A.5: the longest accepted prefix is committed.  At
// temperature 0 the target's choice at node n is am[n] = argmax_v logits[n,v]
// (lowest v on ties).  A non-root node is accepted when its token equals the
// choice at its parent and its parent is accepted.  The deepest accepted node
// wins; equal depths go to the lexicographically smallest root path.
//
// One launch: CTAs stream vocabulary chunks of one row (16-byte loads) and
// fold their (value, index) maximum into a per-row 64-bit key with atomicMax
// (order-preserving float bits in the high word, inverted index in the low
// word, so the lowest index wins ties).  The last CTA to finish a sequence
// (atomic ticket, no waiting) walks that sequence's tree with one warp:
// pointer jumping gives every node its depth, its accepted flag and its
// ancestor set in log2(128) rounds, then a short top-down walk picks the
// lexicographically smallest deepest path.  It resets the keys and the
// ticket so the workspace is ready for the next call.
#include <mutex>

#include "sv_device.cuh"

namespace sv {
namespace acc {

constexpr int kThreads = 256;
constexpr int kChunk = 8192;  // vocabulary entries per CTA (8 float4 per thread)

__device__ __forceinline__ unsigned long long pack_key(float v, int idx) {
  if (v == 0.0f) v = 0.0f;  // -0.0 and +0.0 compare equal
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

__device__ __forceinline__ void take(float v, int i, float& bv, int& bi) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

struct Params {
  const float* logits;
  const int* tokens;
  const int* parents;
  const int* cu_nodes;
  int* argmax_out;
  int* accept_len;
  int* accepted_nodes;
  int* bonus;
  unsigned long long* keys;  // [T]
  int* tickets;              // [B]
  int* err;
  int vocab;
  int batch;
  int chunks;
  int max_depth;
  bool vec4;
};

// Tree walk of sequence b by one warp (N <= 128 nodes, 4 per lane).
__device__ void walk_sequence(const Params& p, int b, int n0, int N) {
  __shared__ int s_am[128], s_par[128], s_ptr[2][128], s_dep[2][128];
  __shared__ uint32_t s_acc[2][128];
  __shared__ uint32_t s_anc[2][128][4];
  const int lane = threadIdx.x & 31;
  if (N < 1 || N > kMaxNodes) {
    report_error(p.err, SV_DEVERR_BAD_TREE);
    if (lane == 0) p.tickets[b] = 0;
    return;
  }

  for (int n = lane; n < N; n += 32) {
    const unsigned long long k = atomicExch(p.keys + n0 + n, 0ull);  // read and reset
    s_am[n] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
    int par = (n == 0) ? -1 : p.parents[n0 + n];
    if (n != 0 && (par < 0 || par >= n)) {
      report_error(p.err, SV_DEVERR_BAD_PARENT);
      par = 0;
    }
    s_par[n] = par;
  }
  __syncwarp();
  for (int n = lane; n < N; n += 32) {
    const int par = s_par[n];
    const bool matched = (n == 0) || (p.tokens[n0 + n] == s_am[par]);
    s_ptr[0][n] = (n == 0) ? 0 : par;
    s_dep[0][n] = (n == 0) ? 0 : 1;
    s_acc[0][n] = matched ? 1u : 0u;
    uint32_t a[4] = {0, 0, 0, 0};
    a[n >> 5] |= 1u << (n & 31);
    if (n != 0) a[par >> 5] |= 1u << (par & 31);
#pragma unroll
    for (int w = 0; w < 4; ++w) s_anc[0][n][w] = a[w];
    if (p.argmax_out != nullptr) p.argmax_out[n0 + n] = s_am[n];
  }
  __syncwarp();
  // pointer jumping: after round r, ptr = 2^(r+1)-th ancestor (clamped at
  // the root), dep = distance to it, acc = all matched on the way, anc =
  // every node within that distance.
  int cur = 0;
  for (int round = 0; round < 7; ++round) {
    const int nxt = cur ^ 1;
    for (int n = lane; n < N; n += 32) {
      const int q = s_ptr[cur][n];
      s_ptr[nxt][n] = s_ptr[cur][q];
      s_dep[nxt][n] = s_dep[cur][n] + s_dep[cur][q];
      s_acc[nxt][n] = s_acc[cur][n] & s_acc[cur][q];
#pragma unroll
      for (int w = 0; w < 4; ++w) s_anc[nxt][n][w] = s_anc[cur][n][w] | s_anc[cur][q][w];
    }
    __syncwarp();
    cur = nxt;
  }
  // deepest accepted depth
  int best = 0;
  for (int n = lane; n < N; n += 32)
    if (s_acc[cur][n]) best = max(best, s_dep[cur][n]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  // nodes lying on some deepest accepted path
  uint32_t good[4] = {0, 0, 0, 0};
  for (int n = lane; n < N; n += 32)
    if (s_acc[cur][n] && s_dep[cur][n] == best) {
#pragma unroll
      for (int w = 0; w < 4; ++w) good[w] |= s_anc[cur][n][w];
    }
#pragma unroll
  for (int w = 0; w < 4; ++w)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) good[w] |= __shfl_xor_sync(0xffffffffu, good[w], o);
  // top-down: smallest-index child on a deepest path, depth by depth
  if (best > p.max_depth) report_error(p.err, SV_DEVERR_DEPTH);
  int* out_path = p.accepted_nodes + static_cast<size_t>(b) * (p.max_depth + 1);
  int node = 0;
  if (lane == 0) out_path[0] = 0;
  for (int d = 1; d <= best; ++d) {
    int pick = 0x7FFFFFFF;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int n = lane + 32 * s;
      const bool c = n < N && n != 0 && s_par[n] == node && ((good[s] >> lane) & 1u);
      const uint32_t bal = __ballot_sync(0xffffffffu, c);
      if (bal != 0 && pick == 0x7FFFFFFF) pick = 32 * s + (__ffs(bal) - 1);
    }
    if (pick == 0x7FFFFFFF) {  // unreachable for a well-formed tree
      report_error(p.err, SV_DEVERR_BAD_TREE);
      best = d - 1;
      break;
    }
    node = pick;
    if (lane == 0 && d <= p.max_depth) out_path[d] = node;
  }
  for (int d = best + 1 + lane; d <= p.max_depth; d += 32) out_path[d] = -1;
  if (lane == 0) {
    p.accept_len[b] = best;
    p.bonus[b] = s_am[node];
    p.tickets[b] = 0;
  }
}

__global__ void __launch_bounds__(kThreads) greedy_accept_kernel(const __grid_constant__ Params p) {
  const int row = blockIdx.y;
  const int chunk = blockIdx.x;
  __shared__ int s_b, s_last;
  __shared__ float s_v[kThreads / 32];
  __shared__ int s_i[kThreads / 32];

  const int lo = chunk * kChunk;
  const int hi = min(p.vocab, lo + kChunk);
  const float* rowp = p.logits + static_cast<size_t>(row) * p.vocab;
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  if (p.vec4) {
    const float4* r4 = reinterpret_cast<const float4*>(rowp);
    float4 v[kChunk / (4 * kThreads)];
#pragma unroll
    for (int u = 0; u < kChunk / (4 * kThreads); ++u) {
      const int e = lo + 4 * (threadIdx.x + u * kThreads);
      v[u] = (e < hi) ? __ldcs(r4 + (e >> 2)) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int u = 0; u < kChunk / (4 * kThreads); ++u) {
      const int e = lo + 4 * (threadIdx.x + u * kThreads);
      if (e < hi) {
        take(v[u].x, e, bv, bi);
        take(v[u].y, e + 1, bv, bi);
        take(v[u].z, e + 2, bv, bi);
        take(v[u].w, e + 3, bv, bi);
      }
    }
  } else {
    for (int e = lo + threadIdx.x; e < hi; e += kThreads) take(rowp[e], e, bv, bi);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    take(ov, oi, bv, bi);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_v[warp] = bv;
    s_i[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) take(s_v[w], s_i[w], bv, bi);
    if (bi != 0x7FFFFFFF) atomicMax(p.keys + row, pack_key(bv, bi));
    // sequence of this row
    int lo_b = 0, hi_b = p.batch;  // cu_nodes[lo_b] <= row < cu_nodes[hi_b]
    while (hi_b - lo_b > 1) {
      const int mid = (lo_b + hi_b) >> 1;
      if (p.cu_nodes[mid] <= row) lo_b = mid;
      else hi_b = mid;
    }
    s_b = lo_b;
    const int n_rows = p.cu_nodes[lo_b + 1] - p.cu_nodes[lo_b];
    __threadfence();
    const int ticket = atomicAdd(p.tickets + lo_b, 1);
    s_last = (ticket == n_rows * p.chunks - 1);
  }
  __syncthreads();
  if (s_last && warp == 0) {
    __threadfence();
    const int b = s_b;
    const int n0 = p.cu_nodes[b];
    const int N = p.cu_nodes[b + 1] - n0;
    walk_sequence(p, b, n0, N);
  }
}

}  // namespace acc
}  // namespace sv

extern "C" {

sv_status sv_greedy_accept_workspace_size(int batch, int total_nodes, size_t* bytes) {
  if (bytes == nullptr || batch < 1 || total_nodes < 0) return SV_ERR_INVALID_ARG;
  *bytes = sv::kWorkspaceHeader + sv::align_up(static_cast<size_t>(total_nodes) * 8, 256) +
           sv::align_up(static_cast<size_t>(batch) * 4, 256);
  return SV_OK;
}

sv_status sv_greedy_accept(const float* logits, int vocab, const int* tokens, const int* parents,
                           const int* cu_nodes, int batch, int total_nodes, int max_nodes, int max_depth,
                           int* argmax_out, int* accept_len, int* accepted_nodes, int* bonus_token,
                           void* workspace, size_t workspace_bytes, sv_stream_t stream) {
  if (!logits || !tokens || !parents || !cu_nodes || !accept_len || !accepted_nodes || !bonus_token)
    return SV_ERR_INVALID_ARG;
  if (vocab < 1 || batch < 1 || total_nodes < 0 || max_nodes < 1 || max_depth < 0) return SV_ERR_INVALID_ARG;
  if (max_nodes > sv::kMaxNodes) return SV_ERR_UNSUPPORTED;
  if (total_nodes > 65535) return SV_ERR_UNSUPPORTED;
  size_t need = 0;
  sv_greedy_accept_workspace_size(batch, total_nodes, &need);
  if (workspace == nullptr || workspace_bytes < need) return SV_ERR_WORKSPACE;
  if (total_nodes == 0) return SV_OK;
  sv::acc::Params p;
  p.logits = logits;
  p.tokens = tokens;
  p.parents = parents;
  p.cu_nodes = cu_nodes;
  p.argmax_out = argmax_out;
  p.accept_len = accept_len;
  p.accepted_nodes = accepted_nodes;
  p.bonus = bonus_token;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.err = reinterpret_cast<int*>(ws);
  p.keys = reinterpret_cast<unsigned long long*>(ws + sv::kWorkspaceHeader);
  p.tickets = reinterpret_cast<int*>(ws + sv::kWorkspaceHeader + sv::align_up(static_cast<size_t>(total_nodes) * 8, 256));
  p.vocab = vocab;
  p.batch = batch;
  p.chunks = (vocab + sv::acc::kChunk - 1) / sv::acc::kChunk;
  p.max_depth = max_depth;
  p.vec4 = (vocab % 4 == 0) && sv::aligned16(logits);
  dim3 grid(p.chunks, total_nodes);
  sv::acc::greedy_accept_kernel<<<grid, sv::acc::kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Greedy acceptance without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they verify a
// draft tree: a serving engine that hands all free device memory to its KV
// pool at start-up, a plugin running inside a host framework that exposes no
// allocator to it, or a decode loop that forbids allocation after warm-up so
// that its memory footprint and latency stay fixed.  For them this variant
// keeps its scratch (the per-row arg-max keys, the per-sequence tickets and
// the error word) in a fixed array of this library's device module, which
// every GPU that loads the library holds until the process exits.
namespace sv {
namespace acc {

constexpr int kStaticMaxNodes = 8192;
constexpr int kStaticMaxBatch = 1024;
constexpr size_t kStaticScratchBytes = kWorkspaceHeader + static_cast<size_t>(kStaticMaxNodes) * 8 +
                                       static_cast<size_t>(kStaticMaxBatch) * 4 + 512;

static __device__ __align__(256) unsigned char g_accept_scratch[kStaticScratchBytes];

// Device address of the scratch array on the current device.  The first call
// on each device resolves it (with that device current) and caches it.
void* static_scratch(sv_status* st) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *st = SV_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || p == nullptr) {
      *st = SV_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  *st = SV_OK;
  return addr[dev];
}

}  // namespace acc
}  // namespace sv

extern "C" sv_status sv_greedy_accept_noalloc(const float* logits, int vocab, const int* tokens, const int* parents,
                                              const int* cu_nodes, int batch, int total_nodes, int max_nodes,
                                              int max_depth, int* argmax_out, int* accept_len, int* accepted_nodes,
                                              int* bonus_token, int* device_error, sv_stream_t stream) {
  using namespace sv::acc;
  if (batch > kStaticMaxBatch || total_nodes > kStaticMaxNodes) return SV_ERR_UNSUPPORTED;
  if (batch < 1 || total_nodes < 0) return SV_ERR_INVALID_ARG;
  sv_status st = SV_OK;
  void* scratch = static_scratch(&st);
  if (st != SV_OK) return st;
  size_t used = 0;
  st = sv_greedy_accept_workspace_size(batch, total_nodes, &used);
  if (st != SV_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // keys, tickets and the error word must start at zero; the array keeps
  // whatever the previous call left there
  if (cudaMemsetAsync(scratch, 0, used, s) != cudaSuccess) return SV_ERR_CUDA;
  st = sv_greedy_accept(logits, vocab, tokens, parents, cu_nodes, batch, total_nodes, max_nodes, max_depth,
                        argmax_out, accept_len, accepted_nodes, bonus_token, scratch, kStaticScratchBytes, stream);
  if (st != SV_OK) return st;
  if (device_error != nullptr &&
      cudaMemcpyAsync(device_error, scratch, sizeof(int), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}
