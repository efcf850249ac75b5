// KV commit of the accepted path (SpecBlock Appendix A.5: the accepted prefix
// is committed before the next iteration; "Dynamic Speculative Decoding",
// Implementation Details: the KV cache must stay consistent with the
// committed tokens).
//
// For each layer, sequence b and j = 0..accept_len[b], slot L_b + j of the
// paged cache receives the K and V of tree node accepted_nodes[b, j] for all
// KV heads: a bit copy in 16-byte vectors.  One CTA per (j, b, layer); CTAs
// with j > accept_len[b] exit at once.  Source (dense tree buffer) and
// destination (paged cache) never overlap, so the copy needs no ordering.
// The launch is a programmatic dependent of the preceding kernel (the
// acceptance, which lets it become resident at once): no launch gap between
// them, and every CTA waits for that kernel's results before reading them.
#include "sv_device.cuh"

namespace sv {
namespace commit {

struct Params {
  const uint4* tree_k;
  const uint4* tree_v;
  uint4* k_cache;
  uint4* v_cache;
  long long tree_layer_stride;   // in uint4 (8 bf16)
  long long cache_layer_stride;  // in uint4
  const int* block_table;
  const int* ctx_lens;
  const int* cu_nodes;
  const int* accepted_nodes;
  const int* accept_len;
  int* new_ctx_lens;
  int* err;
  int num_pages;
  int max_pages_per_seq;
  int max_depth;
  int num_kv_heads;
  int vec_per_head;  // D / 8
  int page_size;
};

__global__ void __launch_bounds__(256) kv_commit_kernel(const __grid_constant__ Params p) {
  const int j = blockIdx.x;
  const int b = blockIdx.y;
  const int layer = blockIdx.z;
  // Launched as a programmatic dependent of the acceptance: the CTAs are
  // resident while it runs and read the accepted path once it has completed.
  griddep_wait();
  // every index this CTA needs, requested in one round (accepted_nodes has
  // max_depth + 1 entries per sequence, one per CTA in x, so the read is in
  // bounds even for positions past the path)
  const int a = p.accept_len[b];
  const int L = p.ctx_lens[b];
  const int n0 = p.cu_nodes[b];
  const int N = p.cu_nodes[b + 1] - n0;
  const int node = p.accepted_nodes[static_cast<size_t>(b) * (p.max_depth + 1) + j];
  if (j > a) return;
  if (a > p.max_depth) {
    // nothing of this sequence is committed, so its length stays L
    if (threadIdx.x == 0) {
      report_error(p.err, SV_DEVERR_DEPTH);
      if (j == 0 && layer == 0 && p.new_ctx_lens != nullptr) p.new_ctx_lens[b] = L;
    }
    return;
  }
  if (j == 0 && layer == 0 && threadIdx.x == 0 && p.new_ctx_lens != nullptr) p.new_ctx_lens[b] = L + a + 1;
  if (node < 0 || node >= N) {
    if (threadIdx.x == 0) report_error(p.err, SV_DEVERR_BAD_PATH);
    return;
  }
  const int slot = L + j;
  const int lp = slot / p.page_size;
  if (lp >= p.max_pages_per_seq) {
    if (threadIdx.x == 0) report_error(p.err, SV_DEVERR_BAD_PAGE);
    return;
  }
  const int phys = p.block_table[static_cast<size_t>(b) * p.max_pages_per_seq + lp];
  if (phys < 0 || phys >= p.num_pages) {
    if (threadIdx.x == 0) report_error(p.err, SV_DEVERR_BAD_PAGE);
    return;
  }
  const int row = slot - lp * p.page_size;
  const int per_kv = p.num_kv_heads * p.vec_per_head;
  const long long src0 = static_cast<long long>(layer) * p.tree_layer_stride +
                         static_cast<long long>(n0 + node) * per_kv;
  const long long dst0 = static_cast<long long>(layer) * p.cache_layer_stride;
  for (int v = threadIdx.x; v < 2 * per_kv; v += blockDim.x) {
    const int which = v >= per_kv;  // 0 = K, 1 = V
    const int rem = v - which * per_kv;
    const int kh = rem / p.vec_per_head;
    const int e = rem - kh * p.vec_per_head;
    const long long dst = dst0 + ((static_cast<long long>(phys) * p.num_kv_heads + kh) * p.page_size + row) *
                                     p.vec_per_head + e;
    const uint4 val = which ? __ldcs(p.tree_v + src0 + rem) : __ldcs(p.tree_k + src0 + rem);
    if (which) p.v_cache[dst] = val;
    else p.k_cache[dst] = val;
  }
}

}  // namespace commit
}  // namespace sv

extern "C" sv_status sv_kv_commit(const void* tree_k, const void* tree_v, long long tree_layer_stride,
                                  void* k_cache, void* v_cache, long long cache_layer_stride, int num_layers,
                                  int num_pages, const int* block_table, int max_pages_per_seq,
                                  const int* ctx_lens, const int* cu_nodes, const int* accepted_nodes,
                                  const int* accept_len, int batch, int max_depth, int num_kv_heads,
                                  int head_dim, int page_size, int* new_ctx_lens, void* workspace,
                                  size_t workspace_bytes, sv_stream_t stream) {
  using namespace sv;
  if (!tree_k || !tree_v || !k_cache || !v_cache || !block_table || !ctx_lens || !cu_nodes || !accepted_nodes ||
      !accept_len)
    return SV_ERR_INVALID_ARG;
  if (num_layers < 1 || num_pages < 1 || max_pages_per_seq < 1 || batch < 1 || max_depth < 0 ||
      num_kv_heads < 1 || page_size < 1)
    return SV_ERR_INVALID_ARG;
  if (head_dim % 8 != 0 || head_dim < 8) return SV_ERR_UNSUPPORTED;
  if (tree_layer_stride % 8 != 0 || cache_layer_stride % 8 != 0 || tree_layer_stride < 0 || cache_layer_stride < 0)
    return SV_ERR_INVALID_ARG;
  if (!aligned16(tree_k) || !aligned16(tree_v) || !aligned16(k_cache) || !aligned16(v_cache))
    return SV_ERR_INVALID_ARG;
  if (new_ctx_lens != nullptr && static_cast<const void*>(new_ctx_lens) == static_cast<const void*>(ctx_lens))
    return SV_ERR_INVALID_ARG;
  if (workspace != nullptr && workspace_bytes < kWorkspaceHeader) return SV_ERR_WORKSPACE;
  if (max_depth + 1 > 65535 || batch > 65535 || num_layers > 65535) return SV_ERR_UNSUPPORTED;
  commit::Params p;
  p.tree_k = static_cast<const uint4*>(tree_k);
  p.tree_v = static_cast<const uint4*>(tree_v);
  p.k_cache = static_cast<uint4*>(k_cache);
  p.v_cache = static_cast<uint4*>(v_cache);
  p.tree_layer_stride = tree_layer_stride / 8;
  p.cache_layer_stride = cache_layer_stride / 8;
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.cu_nodes = cu_nodes;
  p.accepted_nodes = accepted_nodes;
  p.accept_len = accept_len;
  p.new_ctx_lens = new_ctx_lens;
  p.err = static_cast<int*>(workspace);
  p.num_pages = num_pages;
  p.max_pages_per_seq = max_pages_per_seq;
  p.max_depth = max_depth;
  p.num_kv_heads = num_kv_heads;
  p.vec_per_head = head_dim / 8;
  p.page_size = page_size;
  const int per = 2 * num_kv_heads * (head_dim / 8);
  const int threads = per >= 256 ? 256 : ((per + 31) / 32) * 32;
  cudaLaunchConfig_t cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(max_depth + 1, batch, num_layers);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, commit::kv_commit_kernel, p) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}
