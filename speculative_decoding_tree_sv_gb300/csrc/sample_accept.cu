// Stochastic (temperature > 0) acceptance of a verified draft tree.
//
// Speculative sampling (named in SpecPV section 2; Leviathan et al.) applied
// node by node over the token tree, as in SpecInfer's multi-step form: the
// target distribution at node u is p_u = softmax(logits_u / T); the children
// of u, drawn from the draft distribution q_u, are tried in index order
// against a residual R (initially p_u): child c with token x and uniform r is
// accepted when r < min(1, R(x) / q_u(x)) (q_u(x) = 0 accepts), otherwise
// R <- max(R - q_u, 0) / sum(max(R - q_u, 0)) (unchanged when that sum is
// 0).  The walk from the root follows accepted children to a node z, and the
// bonus token is drawn from z's final residual by inverse CDF with z's own
// uniform.  SpecBlock section 4 and SpecPV Appendix E evaluate T = 0.7, 1.0.
//
// Two launches, both on clusters of kCluster CTAs that split the vocabulary:
//   * node_kernel: one cluster per tree node.  Every residual is a function
//     of the logits, q and the normalisers found so far, so a node keeps only
//     its scalars: the max m of logits / T, Z_0 = sum exp(logits / T - m), and
//     for every rejected child the next normaliser Z_j.  Each normaliser is
//     one pass over the vocabulary (the node's rows stay in L2 after the
//     first); the CTAs exchange their partial sums through distributed shared
//     memory and add them in rank order, so every CTA takes the same
//     decisions.  Results: the accepted child (or -1) and the scalars, in the
//     workspace.
//   * walk_kernel: one cluster per sequence.  It follows the accepted children
//     from the root, then draws the bonus at the last node: one coalesced
//     pass stores the residual mass of every 32-entry chunk in shared memory,
//     the cluster adds its slices in rank order, a warp scan over the chunk
//     sums locates the chunk in which the cumulative sum crosses v * total,
//     and a scan inside that chunk the token.
#include <math.h>

#include "sv_device.cuh"

namespace sv {
namespace samp {

constexpr int kCluster = 8;   // CTAs per node / per sequence (one vocabulary slice each)
constexpr int kThreads = 256;      // per-node CTAs (four per SM: one wave for a Llama-sized tree)
constexpr int kWalkThreads = 1024; // per-sequence CTAs
constexpr int kMaxZ = kMaxNodes;  // Z_0 and one normaliser per rejected child
constexpr int kBatch = 16;        // vocabulary entries a thread requests before using them
constexpr int kMaxChunks = 1024;  // 32-entry chunks of one CTA's slice (vocab <= 2^18 per CTA)

struct NodeParams {
  const float* logits;  // [T, V]
  const float* q;       // [T, V]
  const int* tokens;
  const int* parents;
  const int* cu_nodes;
  const float* u_accept;
  int* acc_child;  // [T] local id of the accepted child, -1 if none
  int* nz;         // [T] normalisers stored (1 + rejected children)
  float* mz;       // [T][1 + kMaxZ]: m, Z_0, Z_1, ...
  int* err;
  int vocab;
  int batch;
  float inv_t;
};

struct WalkParams {
  const float* logits;
  const float* q;
  const int* cu_nodes;
  const float* u_bonus;
  const int* acc_child;
  const int* nz;
  const float* mz;
  int* accepted_child_out;  // optional [T]
  int* accept_len;
  int* accepted_nodes;
  int* bonus;
  int* err;
  int vocab;
  int max_depth;
  float inv_t;
};

// ------------------------------------------------------------ cluster helpers

__device__ __forceinline__ void cluster_arrive_wait() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The float at the same shared-memory offset as `local` in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_peer(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Block-wide sum (fixed order), result in every thread.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) s += red[w];
  return s;
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = -INFINITY;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) s = fmaxf(s, red[w]);
  return s;
}

// Cluster-wide sum of one value per CTA, added in rank order (every CTA gets
// the same float).  `slot` alternates between passes so one barrier per
// reduction suffices.
__device__ __forceinline__ float cluster_sum(float mine, float* slots, int& pass) {
  float* slot = slots + (pass & 1);
  ++pass;
  if (threadIdx.x == 0) *slot = mine;
  cluster_arrive_wait();
  float s = 0.f;
#pragma unroll
  for (int r = 0; r < kCluster; ++r) s += ld_peer(slot, r);
  return s;
}

__device__ __forceinline__ float cluster_max(float mine, float* slots, int& pass) {
  float* slot = slots + (pass & 1);
  ++pass;
  if (threadIdx.x == 0) *slot = mine;
  cluster_arrive_wait();
  float s = -INFINITY;
#pragma unroll
  for (int r = 0; r < kCluster; ++r) s = fmaxf(s, ld_peer(slot, r));
  return s;
}

// Residual after j rejections at one vocabulary entry: R_0 = exp(l/T - m)/Z_0,
// R_i = max(R_{i-1} - q, 0) / Z_i (unchanged where Z_i = 0).  `inv` holds
// 1/Z_0, 1/Z_1, ... (0 for a zero sum): two operations per step.
__device__ __forceinline__ float residual(float l, float qv, float inv_t, float m, const float* inv, int j) {
  float r = expf(l * inv_t - m) * inv[0];
  for (int i = 1; i <= j; ++i) {
    const float iz = inv[i];
    r = iz > 0.f ? fmaxf(r - qv, 0.f) * iz : r;
  }
  return r;
}

__device__ __forceinline__ float reciprocal_or_zero(float z) { return z > 0.f ? 1.f / z : 0.f; }

// Sequence holding node t (cu_nodes[b] <= t < cu_nodes[b + 1]), found by one
// warp with a 32-way search: each round the lanes read 32 evenly spaced
// prefix sums of the remaining range at once.  Every lane returns it.
__device__ __forceinline__ int sequence_of_warp(const int* cu_nodes, int batch, int t) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = batch;  // cu_nodes[lo] <= t < cu_nodes[hi]
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int k = lo + lane * step;
    const bool le = k < hi && cu_nodes[k] <= t;
    const uint32_t bal = __ballot_sync(0xffffffffu, le);
    const int last = 31 - __clz(bal);  // lane 0 (k = lo) always qualifies
    lo = lo + last * step;
    hi = min(hi, lo + step);
  }
  return lo;
}

// ------------------------------------------------------------ per node

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    node_kernel(const __grid_constant__ NodeParams p) {
  __shared__ float slots[2];
  __shared__ float red[kThreads / 32];
  __shared__ float s_mz[1 + kMaxZ];  // m, Z_0, Z_1, ...
  __shared__ float s_inv[kMaxZ];     // 1/Z_0, 1/Z_1, ...
  __shared__ int s_kids[kMaxNodes];
  __shared__ int s_nkids, s_n0;
  const uint32_t rank = cluster_ctarank();
  const int t = blockIdx.x / kCluster;  // global node index
  const int V = p.vocab;
  const int lo = static_cast<int>(static_cast<long long>(V) * rank / kCluster);
  const int hi = static_cast<int>(static_cast<long long>(V) * (rank + 1) / kCluster);
  const float* lrow = p.logits + static_cast<size_t>(t) * V;
  const float* qrow = p.q + static_cast<size_t>(t) * V;
  int pass = 0;

  // children of this node, in index order (warp 0: the sequence's parents
  // read at once, then a ballot per 32 nodes)
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int b = sequence_of_warp(p.cu_nodes, p.batch, t);
    const int n0 = p.cu_nodes[b];
    const int N = min(p.cu_nodes[b + 1] - n0, kMaxNodes);
    const int u = t - n0;
    int k = 0;
    for (int c0 = 0; c0 < N; c0 += 32) {
      const int c = c0 + lane;
      const bool kid = c > u && c < N && p.parents[n0 + c] == u;
      const uint32_t bal = __ballot_sync(0xffffffffu, kid);
      if (kid) s_kids[k + __popc(bal & ((1u << lane) - 1u))] = c;
      k += __popc(bal);
    }
    if (lane == 0) {
      s_nkids = k;
      s_n0 = n0;
    }
  }

  // m and Z_0 in one online pass over this CTA's slice (loads issued kBatch
  // at a time): a running maximum and the sum of exponentials relative to
  // it, merged over warps and then over the cluster's ranks in order
  float mt = -INFINITY, st = 0.f;
  for (int x0 = lo + threadIdx.x; x0 < hi; x0 += kThreads * kBatch) {
    float v[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int x = x0 + k * kThreads;
      v[k] = x < hi ? lrow[x] * p.inv_t : -INFINITY;
    }
    float mb = v[0];
#pragma unroll
    for (int k = 1; k < kBatch; ++k) mb = fmaxf(mb, v[k]);
    if (mb > mt) {
      st = (mt == -INFINITY) ? 0.f : st * expf(mt - mb);
      mt = mb;
    }
    if (mt > -INFINITY) {
#pragma unroll
      for (int k = 0; k < kBatch; ++k) st += expf(v[k] - mt);
    }
  }
  const float m = cluster_max(block_max(mt, red), slots, pass);
  const float se = (mt == -INFINITY) ? 0.f : st * expf(mt - m);
  const float z0 = cluster_sum(block_sum(se, red), slots, pass);
  if (threadIdx.x == 0) {
    s_mz[0] = m;
    s_mz[1] = z0;
    s_inv[0] = reciprocal_or_zero(z0);
  }
  __syncthreads();

  // children in order: accept, or one more normaliser
  int accepted = -1, j = 0;
  const int nk = s_nkids;
  for (int i = 0; i < nk; ++i) {
    const int c = s_kids[i];
    const int x = p.tokens[s_n0 + c];
    float a = 0.f;
    if (x >= 0 && x < V) {
      const float qx = qrow[x];
      const float rx = residual(lrow[x], qx, p.inv_t, m, s_inv, j);
      a = (qx <= 0.f) ? 1.f : fminf(1.f, rx / qx);
    } else if (threadIdx.x == 0 && rank == 0) {
      report_error(p.err, SV_DEVERR_BAD_TREE);
    }
    if (p.u_accept[s_n0 + c] < a) {
      accepted = c;
      break;
    }
    if (j + 1 > kMaxZ - 1) break;  // cannot happen: fewer than 128 children
    float sr = 0.f;
    for (int y0 = lo + threadIdx.x; y0 < hi; y0 += kThreads * kBatch) {
      float lv[kBatch], qv[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int y = y0 + k * kThreads;
        lv[k] = y < hi ? lrow[y] : -INFINITY;  // exp(-inf) = 0: no mass
        qv[k] = y < hi ? qrow[y] : 0.f;
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) sr += fmaxf(residual(lv[k], qv[k], p.inv_t, m, s_inv, j) - qv[k], 0.f);
    }
    const float zj = cluster_sum(block_sum(sr, red), slots, pass);
    ++j;
    if (threadIdx.x == 0) {
      s_mz[1 + j] = zj;
      s_inv[j] = reciprocal_or_zero(zj);
    }
    __syncthreads();
  }
  if (rank == 0 && threadIdx.x == 0) {
    p.acc_child[t] = accepted;
    p.nz[t] = 1 + j;
  }
  if (rank == 0)
    for (int i = threadIdx.x; i < 2 + j; i += kThreads) p.mz[static_cast<size_t>(t) * (1 + kMaxZ) + i] = s_mz[i];
  cluster_arrive_wait();  // no CTA leaves while a peer may still read its slots
}

// ------------------------------------------------------------ per sequence

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kWalkThreads)
    walk_kernel(const __grid_constant__ WalkParams p) {
  // a following KV commit may become resident now (it waits for completion)
  griddep_launch_dependents();
  __shared__ float slots[3];  // this CTA's residual total, found token, last token with mass
  __shared__ float s_mz[1 + kMaxZ];
  __shared__ float s_inv[kMaxZ];
  __shared__ int s_path[kMaxNodes];
  __shared__ int s_len, s_z;
  __shared__ float s_chunk[kMaxChunks];  // residual mass of each 32-entry chunk of this CTA's slice
  __shared__ int s_last[kWalkThreads / 32];
  __shared__ float s_run;
  __shared__ int s_hit;
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x / kCluster;
  const int n0 = p.cu_nodes[b];
  const int N = p.cu_nodes[b + 1] - n0;
  const int V = p.vocab;

  // the walk (thread 0 of every CTA: the same result everywhere), over the
  // sequence's accepted children staged in shared memory
  __shared__ int s_acc[kMaxNodes];
  for (int i = threadIdx.x; i < N && i < kMaxNodes; i += kWalkThreads) s_acc[i] = p.acc_child[n0 + i];
  __syncthreads();
  if (threadIdx.x == 0) {
    int z = 0, len = 0;
    s_path[0] = 0;
    if (N >= 1 && N <= kMaxNodes) {
      for (int step = 0; step < N; ++step) {
        const int c = s_acc[z];
        if (c <= z || c >= N) break;  // -1 (none); a child always has a larger index
        z = c;
        s_path[++len] = z;
      }
    } else if (rank == 0) {
      report_error(p.err, SV_DEVERR_BAD_TREE);
    }
    s_len = len;
    s_z = z;
  }
  __syncthreads();
  if (N < 1 || N > kMaxNodes) {
    // no valid tree (reported above): nothing to draw from; every CTA of the
    // cluster leaves here, before any cluster barrier
    if (rank == 0 && threadIdx.x == 0) {
      int* out_path = p.accepted_nodes + static_cast<size_t>(b) * (p.max_depth + 1);
      for (int d = 0; d <= p.max_depth; ++d) out_path[d] = -1;
      p.accept_len[b] = 0;
      p.bonus[b] = -1;
    }
    return;
  }
  const int z = s_z;
  const int t = n0 + z;
  const int nz = max(1, min(p.nz[t], kMaxZ));
  for (int i = threadIdx.x; i < 1 + nz; i += kWalkThreads) {
    const float v = p.mz[static_cast<size_t>(t) * (1 + kMaxZ) + i];
    s_mz[i] = v;
    if (i >= 1) s_inv[i - 1] = reciprocal_or_zero(v);
  }
  __syncthreads();
  const int j = nz - 1;  // normalisers beyond Z_0
  const float m = s_mz[0];
  const float* lrow = p.logits + static_cast<size_t>(t) * V;
  const float* qrow = p.q + static_cast<size_t>(t) * V;
  const int lo = static_cast<int>(static_cast<long long>(V) * rank / kCluster);
  const int hi = static_cast<int>(static_cast<long long>(V) * (rank + 1) / kCluster);
  const int nchunks = (hi - lo + 31) / 32;

  // pass 1: the residual mass of every 32-entry chunk (a warp takes chunks
  // w, w + 8, ...; kBatch chunks' loads in flight per lane), and the last
  // entry with mass
  int last = -1;
  for (int c0 = warp; c0 < nchunks; c0 += (kWalkThreads / 32) * kBatch) {
    float lv[kBatch], qv[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int x = lo + (c0 + k * (kWalkThreads / 32)) * 32 + lane;
      lv[k] = x < hi ? lrow[x] : -INFINITY;
      qv[k] = (x < hi && j > 0) ? qrow[x] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int c = c0 + k * (kWalkThreads / 32);
      float r = residual(lv[k], qv[k], p.inv_t, m, s_inv, j);
      if (r > 0.f) last = max(last, lo + c * 32 + lane);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
      if (lane == 0 && c < nchunks) s_chunk[c] = r;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  if (lane == 0) s_last[warp] = last;
  __syncthreads();
  // this slice's mass: warp 0, a lane per run of consecutive chunks, an
  // inclusive scan over the lanes (kept for the search below)
  const int per = (nchunks + 31) / 32;
  const int q0 = min(nchunks, lane * per), q1 = min(nchunks, q0 + per);
  float run_mass = 0.f, run_incl = 0.f;
  if (warp == 0) {
    for (int c = q0; c < q1; ++c) run_mass += s_chunk[c];
    run_incl = run_mass;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, run_incl, o);
      if (lane >= o) run_incl += y;
    }
    const float tot = __shfl_sync(0xffffffffu, run_incl, 31);
    if (lane == 0) {
      int l = -1;
      for (int w = 0; w < kWalkThreads / 32; ++w) l = max(l, s_last[w]);
      slots[0] = tot;
      slots[2] = static_cast<float>(l);  // exact: tokens are below 2^24
    }
  }
  cluster_arrive_wait();
  // every rank adds the slices' masses in the same order, so the ranges
  // [before, before + mine) partition [0, total) identically everywhere; the
  // last rank also owns a target at or above the total (rounding)
  float before = 0.f, total = 0.f, mine_rank = 0.f;
  for (int r = 0; r < kCluster; ++r) {  // ranks in order
    const float v = ld_peer(&slots[0], r);
    if (r < static_cast<int>(rank)) before += v;
    if (r == static_cast<int>(rank)) mine_rank = v;
    total += v;
  }
  const float target = p.u_bonus[t] * total;
  const bool own = (target >= before && target < before + mine_rank) ||
                   (rank == kCluster - 1 && target >= before + mine_rank);

  // the chunk where the running sum first exceeds the target (one warp: a
  // lane per run of chunks, an exclusive scan over the lanes), then the
  // entry inside it
  if (warp == 0 && !own && lane == 0) slots[1] = -1.f;
  if (warp == 0 && own) {
    const float mine = run_mass;
    const float excl = before + (run_incl - mine);
    const bool here = excl <= target && excl + mine > target;
    const uint32_t bal = __ballot_sync(0xffffffffu, here);
    if (lane == 0) s_hit = -1;
    __syncwarp();
    if (bal != 0 && lane == __ffs(bal) - 1) {
      float run = excl;
      int hit = q1 - 1;
      for (int c = q0; c < q1; ++c) {
        if (run + s_chunk[c] > target) {
          hit = c;
          break;
        }
        run += s_chunk[c];
      }
      s_hit = hit;
      s_run = run;
    } else if (bal == 0 && lane == 0) {
      // the scan's rounding put the target past this slice's end: its last
      // chunk with mass
      int hit = -1;
      for (int c = nchunks - 1; c >= 0 && hit < 0; --c)
        if (s_chunk[c] > 0.f) hit = c;
      float run = before;
      for (int c = 0; c < hit; ++c) run += s_chunk[c];
      s_hit = hit;
      s_run = run;
    }
    __syncwarp();
    const int hit = s_hit;
    float found = -1.f;
    if (hit >= 0) {
      const int x = lo + hit * 32 + lane;
      const float r = x < hi ? residual(lrow[x], j > 0 ? qrow[x] : 0.f, p.inv_t, m, s_inv, j) : 0.f;
      float in = r;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, in, o);
        if (lane >= o) in += y;
      }
      const uint32_t cross = __ballot_sync(0xffffffffu, x < hi && s_run + in > target);
      // rounding between the chunk's two sums: the chunk's last entry with mass
      const uint32_t mass = __ballot_sync(0xffffffffu, x < hi && r > 0.f);
      const int pick = cross != 0 ? __ffs(cross) - 1 : (mass != 0 ? 31 - __clz(mass) : -1);
      if (pick >= 0) found = static_cast<float>(lo + hit * 32 + pick);
    }
    if (lane == 0) slots[1] = found;
  }
  cluster_arrive_wait();
  // the lowest rank that found the crossing; if none did (the uniform at the
  // very top after rounding), the last token with mass
  int token = -1, fallback = -1;
  for (int r = 0; r < kCluster; ++r) {
    const float f = ld_peer(&slots[1], r);
    if (token < 0 && f >= 0.f) token = static_cast<int>(f);
    fallback = max(fallback, static_cast<int>(ld_peer(&slots[2], r)));
  }
  if (token < 0) token = fallback >= 0 ? fallback : V - 1;
  if (rank == 0 && threadIdx.x == 0) {
    const int len = s_len;
    if (len > p.max_depth) report_error(p.err, SV_DEVERR_DEPTH);
    int* out_path = p.accepted_nodes + static_cast<size_t>(b) * (p.max_depth + 1);
    for (int d = 0; d <= p.max_depth; ++d) out_path[d] = d <= len ? s_path[d] : -1;
    p.accept_len[b] = len;
    p.bonus[b] = token;
  }
  if (p.accepted_child_out != nullptr && rank == 0)
    for (int i = threadIdx.x; i < N && i < kMaxNodes; i += kWalkThreads) p.accepted_child_out[n0 + i] = s_acc[i];
  cluster_arrive_wait();  // no CTA leaves while a peer may still read its slots
}

}  // namespace samp
}  // namespace sv

extern "C" {

sv_status sv_sample_accept_workspace_size(int batch, int total_nodes, size_t* bytes) {
  if (bytes == nullptr || batch < 1 || total_nodes < 0) return SV_ERR_INVALID_ARG;
  const size_t T = static_cast<size_t>(total_nodes);
  *bytes = sv::kWorkspaceHeader + 2 * sv::align_up(T * 4, 256) +
           sv::align_up(T * (1 + sv::samp::kMaxZ) * sizeof(float), 256);
  return SV_OK;
}

sv_status sv_sample_accept(const float* logits, const float* draft_probs, int vocab, float temperature,
                           const int* tokens, const int* parents, const int* cu_nodes, int batch, int total_nodes,
                           int max_nodes, int max_depth, const float* u_accept, const float* u_bonus,
                           int* accepted_child, int* accept_len, int* accepted_nodes, int* bonus_token,
                           void* workspace, size_t workspace_bytes, sv_stream_t stream) {
  using namespace sv::samp;
  if (!logits || !draft_probs || !tokens || !parents || !cu_nodes || !u_accept || !u_bonus || !accept_len ||
      !accepted_nodes || !bonus_token)
    return SV_ERR_INVALID_ARG;
  if (vocab < kCluster || batch < 1 || total_nodes < 0 || max_nodes < 1 || max_depth < 0) return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (max_nodes > sv::kMaxNodes || vocab > kCluster * kMaxChunks * 32) return SV_ERR_UNSUPPORTED;
  size_t need = 0;
  sv_sample_accept_workspace_size(batch, total_nodes, &need);
  if (workspace == nullptr || workspace_bytes < need) return SV_ERR_WORKSPACE;
  if (total_nodes == 0) return SV_OK;
  if (static_cast<long long>(total_nodes) * kCluster > 0x7FFFFFFFll || static_cast<long long>(batch) * kCluster > 0x7FFFFFFFll)
    return SV_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t T = static_cast<size_t>(total_nodes);
  int* acc = reinterpret_cast<int*>(ws + sv::kWorkspaceHeader);
  int* nz = reinterpret_cast<int*>(ws + sv::kWorkspaceHeader + sv::align_up(T * 4, 256));
  float* mz = reinterpret_cast<float*>(ws + sv::kWorkspaceHeader + 2 * sv::align_up(T * 4, 256));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  NodeParams np;
  np.logits = logits;
  np.q = draft_probs;
  np.tokens = tokens;
  np.parents = parents;
  np.cu_nodes = cu_nodes;
  np.u_accept = u_accept;
  np.acc_child = acc;
  np.nz = nz;
  np.mz = mz;
  np.err = reinterpret_cast<int*>(ws);
  np.vocab = vocab;
  np.batch = batch;
  np.inv_t = 1.0f / temperature;
  node_kernel<<<total_nodes * kCluster, kThreads, 0, s>>>(np);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  WalkParams wp;
  wp.logits = logits;
  wp.q = draft_probs;
  wp.cu_nodes = cu_nodes;
  wp.u_bonus = u_bonus;
  wp.acc_child = acc;
  wp.nz = nz;
  wp.mz = mz;
  wp.accepted_child_out = accepted_child;
  wp.accept_len = accept_len;
  wp.accepted_nodes = accepted_nodes;
  wp.bonus = bonus_token;
  wp.err = reinterpret_cast<int*>(ws);
  wp.vocab = vocab;
  wp.max_depth = max_depth;
  wp.inv_t = np.inv_t;
  walk_kernel<<<batch * kCluster, kWalkThreads, 0, s>>>(wp);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

}  // extern "C"
