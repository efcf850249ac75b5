// Greedy (temperature 0) acceptance of a verified draft tree.
//
// SpecBlock Appendix A.5: the longest accepted prefix is committed.  At
// temperature 0 the target's choice at node n is am[n] = argmax_v logits[n,v]
// (lowest v on ties).  A non-root node is accepted when its token equals the
// choice at its parent and its parent is accepted.  The deepest accepted node
// wins; equal depths go to the lexicographically smallest root path.
//
// One launch, one CTA per (16384-entry vocabulary chunk, row).  A CTA asks
// for its whole chunk at once: the first half with 16-byte asynchronous
// copies into shared memory (cp.async), the second half with 16-byte loads
// into registers.  Holding half of the chunk in shared memory keeps the
// registers per thread low enough that every CTA of a Llama-sized step
// (60 rows x 8 chunks) is resident, so the whole logits tensor is in flight
// in one wave; for larger steps each SM keeps five CTAs' 64 KB in flight.  The CTA
// folds its (value, index) maximum into a per-row 64-bit key with atomicMax
// (order-preserving float bits in the high word, inverted index in the low
// word, so the lowest index wins ties).  The last CTA to finish a sequence
// (atomic ticket, no waiting) walks that sequence's tree: its threads load
// one node each, then one warp (four nodes per lane, warp syncs only) jumps
// pointers, which gives every node its depth, its accepted flag and its
// ancestor set in at most log2(128) rounds, and a short top-down walk picks
// the lexicographically smallest deepest path.  It
// resets the keys and the ticket so the workspace is ready for the next call.
//
// Rows that do not start on a 16-byte boundary (vocabulary not a multiple of
// 4, or an unaligned logits pointer) are read with plain loads.
#include <mutex>

#include "sv_device.cuh"

namespace sv {
namespace acc {

constexpr int kThreads = 256;
constexpr int kSmemPart = 8192;  // entries copied into shared memory (8 x 16 B per thread)
constexpr int kRegPart = 8192;   // entries loaded into registers (8 float4 per thread)
constexpr int kChunk = kSmemPart + kRegPart;
constexpr uint32_t kDynSmem = kSmemPart * 4;  // the shared-memory part, later the tree walk's arrays

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

// Outputs of a sequence whose tree cannot be walked (no node, or more than
// kMaxNodes): accept length 0, no bonus token (-1), a path of -1; the error
// word records SV_DEVERR_BAD_TREE.  Called by every thread of a CTA.
__device__ void write_no_tree(const Params& p, int b) {
  int* out_path = p.accepted_nodes + static_cast<size_t>(b) * (p.max_depth + 1);
  for (int d = threadIdx.x; d <= p.max_depth; d += blockDim.x) out_path[d] = -1;
  if (threadIdx.x == 0) {
    p.accept_len[b] = 0;
    p.bonus[b] = -1;
    report_error(p.err, SV_DEVERR_BAD_TREE);
  }
}

// Tree walk of sequence b (nodes n0 .. n0 + N - 1): the CTA loads the nodes
// (one per thread), then one warp jumps pointers and walks; `scratch` is 8 KB
// of shared memory nothing else uses now.
__device__ void walk_sequence(const Params& p, int b, int n0, int N, uint8_t* scratch) {
  int* s_am = reinterpret_cast<int*>(scratch);                  // [128]
  int* s_par = s_am + kMaxNodes;                                // [128]
  int* s_ptr = s_par + kMaxNodes;                               // [2][128]
  int* s_dep = s_ptr + 2 * kMaxNodes;                           // [2][128]
  uint32_t* s_acc = reinterpret_cast<uint32_t*>(s_dep + 2 * kMaxNodes);  // [2][128]
  uint32_t* s_anc = s_acc + 2 * kMaxNodes;                      // [2][128][4]
  const int t = threadIdx.x;
  if (N < 1 || N > kMaxNodes) {  // uniform over the CTA
    // no walk: the keys go back to zero for the next call on this
    // workspace, and the sequence gets defined outputs
    for (int i = t; i < N; i += blockDim.x) p.keys[n0 + i] = 0ull;
    write_no_tree(p, b);
    if (t == 0) p.tickets[b] = 0;
    return;
  }
  int am = 0, par = -1, tok = 0;
  if (t < N) {
    // the keys were last written by atomics at L2: read them there, then reset
    const unsigned long long k = __ldcg(p.keys + n0 + t);
    p.keys[n0 + t] = 0ull;
    am = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
    if (t != 0) {
      par = p.parents[n0 + t];
      tok = p.tokens[n0 + t];
      if (par < 0 || par >= t) {
        report_error(p.err, SV_DEVERR_BAD_PARENT);
        par = 0;
      }
    }
    s_am[t] = am;
    s_par[t] = par;
  }
  __syncthreads();
  if (t < N) {
    const bool matched = (t == 0) || (tok == s_am[par]);
    s_ptr[t] = (t == 0) ? 0 : par;
    s_dep[t] = (t == 0) ? 0 : 1;
    s_acc[t] = matched ? 1u : 0u;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t a = ((t >> 5) == w) ? (1u << (t & 31)) : 0u;
      if (t != 0 && (par >> 5) == w) a |= 1u << (par & 31);
      s_anc[t * 4 + w] = a;
    }
    if (p.argmax_out != nullptr) p.argmax_out[n0 + t] = am;
  }
  __syncthreads();
  if (t >= 32) return;
  // The rest is one warp's (lane owns nodes lane + 32 s): warp syncs instead
  // of block barriers keep each round a few hundred cycles shorter.
  const int lane = t;
  // pointer jumping: after round r, ptr = 2^(r+1)-th ancestor (clamped at
  // the root), dep = distance to it, acc = all matched on the way, anc =
  // every node within that distance; done once every pointer is the root
  int cur = 0;
  for (int round = 0;; ++round) {
    bool mine = true;
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
      const int n = lane + 32 * sl;
      if (n < N && s_ptr[cur * kMaxNodes + n] != 0) mine = false;
    }
    if (__all_sync(0xffffffffu, mine) || round == 7) break;
    const int nxt = cur ^ 1;
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
      const int n = lane + 32 * sl;
      if (n < N) {
        const int q = s_ptr[cur * kMaxNodes + n];
        s_ptr[nxt * kMaxNodes + n] = s_ptr[cur * kMaxNodes + q];
        s_dep[nxt * kMaxNodes + n] = s_dep[cur * kMaxNodes + n] + s_dep[cur * kMaxNodes + q];
        s_acc[nxt * kMaxNodes + n] = s_acc[cur * kMaxNodes + n] & s_acc[cur * kMaxNodes + q];
#pragma unroll
        for (int w = 0; w < 4; ++w)
          s_anc[(nxt * kMaxNodes + n) * 4 + w] = s_anc[(cur * kMaxNodes + n) * 4 + w] | s_anc[(cur * kMaxNodes + q) * 4 + w];
      }
    }
    __syncwarp();
    cur = nxt;
  }
  // deepest accepted depth, then the nodes lying on some deepest accepted path
  bool acc_n[4];
  int dep_n[4], par_n[4];
  int best = 0;
#pragma unroll
  for (int sl = 0; sl < 4; ++sl) {
    const int n = lane + 32 * sl;
    acc_n[sl] = n < N && s_acc[cur * kMaxNodes + n] != 0u;
    dep_n[sl] = acc_n[sl] ? s_dep[cur * kMaxNodes + n] : 0;
    par_n[sl] = n < N ? s_par[n] : -1;
    best = max(best, dep_n[sl]);
  }
  best = __reduce_max_sync(0xffffffffu, best);
  uint32_t good[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int sl = 0; sl < 4; ++sl) {
    const int n = lane + 32 * sl;
    if (acc_n[sl] && dep_n[sl] == best) {
#pragma unroll
      for (int w = 0; w < 4; ++w) good[w] |= s_anc[(cur * kMaxNodes + n) * 4 + w];
    }
  }
#pragma unroll
  for (int w = 0; w < 4; ++w) good[w] = __reduce_or_sync(0xffffffffu, good[w]);
  // top-down: smallest-index child on a deepest path, depth by depth
  if (lane == 0 && best > p.max_depth) report_error(p.err, SV_DEVERR_DEPTH);
  int* out_path = p.accepted_nodes + static_cast<size_t>(b) * (p.max_depth + 1);
  int node = 0, len = best;
  if (lane == 0) out_path[0] = 0;
  for (int d = 1; d <= best; ++d) {
    int pick = 0x7FFFFFFF;
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
      const int n = lane + 32 * sl;
      const bool c = n < N && n != 0 && par_n[sl] == node && ((good[sl] >> lane) & 1u);
      const uint32_t bal = __ballot_sync(0xffffffffu, c);
      if (bal != 0 && pick == 0x7FFFFFFF) pick = 32 * sl + (__ffs(bal) - 1);
    }
    if (pick == 0x7FFFFFFF) {  // unreachable for a well-formed tree
      if (lane == 0) report_error(p.err, SV_DEVERR_BAD_TREE);
      len = d - 1;
      break;
    }
    node = pick;
    if (lane == 0 && d <= p.max_depth) out_path[d] = node;
  }
  for (int d = len + 1 + lane; d <= p.max_depth; d += 32) out_path[d] = -1;
  if (lane == 0) {
    p.accept_len[b] = len;
    p.bonus[b] = s_am[node];
    p.tickets[b] = 0;
  }
}

__global__ void __launch_bounds__(kThreads) greedy_accept_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t dyn[];  // [kSmemPart] floats, then the walk's arrays
  // A following KV commit (launched as a programmatic dependent) may become
  // resident now; it waits for this grid to complete before reading the path.
  griddep_launch_dependents();
  __shared__ int s_b, s_n0, s_n, s_last;
  __shared__ float s_v[kThreads / 32];
  __shared__ int s_i[kThreads / 32];
  const int row = blockIdx.y;
  const int chunk = blockIdx.x;
  const int lo = chunk * kChunk;
  const int hi = min(p.vocab, lo + kChunk);
  const int smem_hi = min(hi, lo + kSmemPart);  // shared-memory part [lo, smem_hi), registers [lo + kSmemPart, hi)
  const float* rowp = p.logits + static_cast<size_t>(row) * p.vocab;
  const int n4s = (smem_hi - lo) >> 2;  // float4 of the shared-memory part
  if (p.vec4) {
#pragma unroll
    for (int u = 0; u < kSmemPart / (4 * kThreads); ++u) {
      const int j = threadIdx.x + u * kThreads;
      if (j < n4s)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dyn + 16 * j)),
                     "l"(rowp + lo + 4 * j) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  if (p.vec4) {
    const float4* r4 = reinterpret_cast<const float4*>(rowp);
    float4 v[kRegPart / (4 * kThreads)];
#pragma unroll
    for (int u = 0; u < kRegPart / (4 * kThreads); ++u) {
      const int e = lo + kSmemPart + 4 * (threadIdx.x + u * kThreads);
      v[u] = (e < hi) ? __ldcs(r4 + (e >> 2)) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int u = 0; u < kRegPart / (4 * kThreads); ++u) {
      const int e = lo + kSmemPart + 4 * (threadIdx.x + u * kThreads);
      if (e < hi) {
        take(v[u].x, e, bv, bi);
        take(v[u].y, e + 1, bv, bi);
        take(v[u].z, e + 2, bv, bi);
        take(v[u].w, e + 3, bv, bi);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();  // every thread's copies have landed
    const float4* b4 = reinterpret_cast<const float4*>(dyn);
#pragma unroll
    for (int u = 0; u < kSmemPart / (4 * kThreads); ++u) {
      const int j = threadIdx.x + u * kThreads;
      if (j < n4s) {
        const float4 w = b4[j];
        const int e = lo + 4 * j;
        take(w.x, e, bv, bi);
        take(w.y, e + 1, bv, bi);
        take(w.z, e + 2, bv, bi);
        take(w.w, e + 3, bv, bi);
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
    const int n0 = p.cu_nodes[lo_b];
    const int n_rows = p.cu_nodes[lo_b + 1] - n0;
    s_b = lo_b;
    s_n0 = n0;
    s_n = n_rows;
    __threadfence();
    const int ticket = atomicAdd(p.tickets + lo_b, 1);
    s_last = (ticket == n_rows * p.chunks - 1);
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    walk_sequence(p, s_b, s_n0, s_n, dyn);
  }
  // A sequence without nodes owns no row, so no CTA above is its last one:
  // the first CTA gives every such sequence its defined outputs.
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int b0 = 0; b0 < p.batch; b0 += kThreads) {
      const int bb = b0 + threadIdx.x;
      const bool empty = bb < p.batch && p.cu_nodes[bb + 1] - p.cu_nodes[bb] < 1;
      const int n_empty = __syncthreads_count(empty);
      if (n_empty == 0) continue;
      __shared__ int s_empty[kThreads];
      __shared__ int s_count;
      if (threadIdx.x == 0) s_count = 0;
      __syncthreads();
      if (empty) s_empty[atomicAdd(&s_count, 1)] = bb;
      __syncthreads();
      for (int i = 0; i < n_empty; ++i) write_no_tree(p, s_empty[i]);
      __syncthreads();
    }
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
  sv::acc::greedy_accept_kernel<<<grid, sv::acc::kThreads, sv::acc::kDynSmem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
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

// Unique id (over the process) of the context current on this thread, 0 when
// it cannot be read.  A cudaDeviceReset ends a device's primary context; the
// next one gets a new id and this library's module is loaded into it afresh.
unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static std::once_flag once;
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(fn);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch array on the current device.  The first call
// on each device resolves it (with that device current) and caches it with
// the id of the device's context; a later call in another context of that
// device (after a cudaDeviceReset) resolves it again.
void* static_scratch(sv_status* st) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  static unsigned long long ctx_id[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *st = SV_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long id = current_context_id();
  if (addr[dev] == nullptr || id == 0 || id != ctx_id[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || p == nullptr) {
      *st = SV_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
    ctx_id[dev] = current_context_id();
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
