/*
 * sv.h — C ABI of the GB300 (sm_103a) tree-verification library (libsv.so).
 *
 * Speculative decoding drafts a tree of candidate tokens and has the target
 * model score every node in one forward pass, then commits the longest
 * accepted prefix (SpecBlock, Appendix A.5 "Inference procedure"; SpecPV,
 * section 1 and section 3.2).  This library implements the data-parallel
 * hot path of that verification step:
 *
 *   sv_tree_attention  tree-masked, paged GQA attention of all tree nodes
 *                      against the context KV cache (full, or a SpecPV
 *                      partial page list), one layer per call;
 *   sv_greedy_accept   per-node vocabulary arg-max and the longest accepted
 *                      root path (temperature 0);
 *   sv_sample_accept   speculative sampling over the tree (temperature > 0);
 *   sv_kv_commit       copy of the accepted path's K/V into the paged cache
 *                      for every layer.
 *
 * Conventions shared by every entry point
 *   - All pointers not marked "host" are device pointers.  The caller owns
 *     all memory; the library allocates nothing.
 *   - Every call is asynchronous on the given stream and performs no host
 *     synchronisation (sv_get_device_error excepted).
 *   - Host-checkable errors (null pointers, unsupported shapes, misaligned
 *     pointers, workspace too small) return synchronously without launching
 *     anything.  Launch failures return SV_ERR_CUDA.
 *   - Device-resident index data (block tables, parents, page lists, paths)
 *     is range-checked by the kernels: an out-of-range value is skipped and
 *     recorded as a nonzero code in the workspace's error word, never as a
 *     trap.  Read it with sv_get_device_error.
 *   - bf16 tensors are IEEE bfloat16, little endian, rows contiguous, and
 *     must start on 16-byte boundaries.  Inputs are finite; NaN is
 *     unsupported.
 *   - A workspace must be zero-filled once after allocation (for example with
 *     cudaMemset) and must not be shared by calls that may run concurrently.
 *     Each call leaves its workspace ready for the next call; after a call
 *     that reported a device error or a timeout, zero it again.
 *   - Symbols are thread-safe; per-stream ordering is the caller's.
 */
#ifndef SV_H_
#define SV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* sv_stream_t;

typedef enum sv_status {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer   */
  SV_ERR_UNSUPPORTED = 2,  /* shape outside the supported set             */
  SV_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed */
  SV_ERR_WORKSPACE = 4,    /* workspace missing or too small              */
  SV_ERR_DEVICE = 5,       /* the device error word holds a nonzero code  */
  SV_ERR_TIMEOUT = 6       /* a bounded device-side wait ran out          */
} sv_status;

/* Codes a kernel writes into the workspace's error word (first 4 bytes). */
enum {
  SV_DEVERR_NONE = 0,
  SV_DEVERR_TIMEOUT = 1,     /* a bounded wait in a kernel ran out          */
  SV_DEVERR_BAD_PARENT = 2,  /* parent[i] not in [0, i) for a non-root node */
  SV_DEVERR_BAD_PAGE = 3,    /* page id outside [0, num_pages) or table     */
  SV_DEVERR_BAD_PATH = 4,    /* accepted path node outside its tree         */
  SV_DEVERR_DEPTH = 5,       /* accepted depth exceeds max_depth            */
  SV_DEVERR_BAD_TREE = 6     /* a tree has no nodes or more than max_nodes  */
};

/* Library ABI version (incremented on incompatible changes). */
int sv_abi_version(void);

/* Static, human-readable name of a status code. */
const char* sv_status_string(sv_status status);

/* ------------------------------------------------------------------------
 * Tree-verification attention (one layer).
 *
 * Defined by: SpecBlock Appendix A.5 (all drafted positions scored in one
 * parallel target forward); SpecBlock Appendix A.2 (a position sees the
 * verified prefix and its on-path predecessors, off-path positions are
 * masked); SpecPV section 3.2 (partial verification: the retained sink,
 * retrieved, window and buffer blocks form one continuous KV segment).
 *
 * For sequence b with N_b tree nodes and context length L_b, node i of the
 * tree (sequence-local index; node 0 is the root, the last accepted token)
 * and query head h (KV head h / G, G = Hq / Hkv) computes
 *     out[i,h] = sum_j softmax_j(scale * q[i,h] . k_j) v_j
 * over the keys j = the context tokens (all of 0..L_b-1, or the tokens of
 * the listed pages in list order) followed by the tree nodes that are
 * ancestors of i or i itself.  The root is not part of L_b.  Q and K arrive
 * with positional encoding already applied.
 * ---------------------------------------------------------------------- */
/* Options of sv_tree_attention (sv_attn_params.flags).
 *
 * SV_ATTN_EARLY_CONTEXT: the kernel is launched as a programmatic dependent
 * of the kernel before it in the stream, so it may start while that kernel
 * is still running; by default it reads nothing before that kernel has
 * finished.  With this flag it already reads the page tables, ctx_lens,
 * cu_nodes, parents, the partial page list and the context K/V pages (cache
 * slots below ctx_lens[b]) in that window, and waits only before it reads Q
 * and the tree's K/V and before it writes anything.  Set it when none of
 * those inputs is written by a preceding kernel that signals early
 * completion (griddepcontrol.launch_dependents) before writing them; the
 * kernels of this library never write them.  Consecutive layers then
 * overlap one layer's context loads with the previous layer's tail. */
enum sv_attn_flags {
  SV_ATTN_EARLY_CONTEXT = 1,
  /* Kernel choice (at most one; by default a cost model picks).  PAIRED: one
   * CTA per 128-row tile, the two row tiles of a group share each K/V tile
   * by cluster multicast, scores double-buffered in TMEM; suits short
   * contexts split across many CTAs.  WIDE: one CTA per 256-row group, each
   * K/V tile staged in one SM only, the context split evenly per group.
   * DEALT: the WIDE engine in one CTA per SM (a multiple of Hkv), groups of
   * one CTA per KV head taking equal contiguous ranges of the call's
   * (sequence, row group, tile) work, so batches of uneven or many
   * sequences run in one even wave. */
  SV_ATTN_KERNEL_PAIRED = 2,
  SV_ATTN_KERNEL_WIDE = 4,
  SV_ATTN_KERNEL_DEALT = 8
};

typedef struct sv_attn_params {
  /* shapes (host values) */
  int batch;              /* B, 1..65535                                     */
  int num_q_heads;        /* Hq                                              */
  int num_kv_heads;       /* Hkv; G = Hq / Hkv must be 1, 2, 4, 8 or 16     */
  int head_dim;           /* D: 64 or 128                                    */
  int page_size;          /* tokens per KV page: 16                          */
  int num_pages;          /* pages in this layer's pool (cache dim 0)        */
  int total_nodes;        /* T = cu_nodes[B] (host copy)                     */
  int max_nodes;          /* max_b N_b (host copy), 1..128                   */
  int max_pages_per_seq;  /* row length of block_table                       */
  int max_kv_pages;       /* partial mode: max_b listed pages (host copy)    */
  int num_splits;         /* KV splits per (sequence, head group); 0 = auto
                             (a count > 0 selects a split kernel, paired or
                             wide, unless SV_ATTN_KERNEL_DEALT is set; the
                             dealt kernel ignores it)                        */
  int split_reduce;       /* how splits merge: 0 = auto, 2 = through
                             workspace partials and a combine kernel (the
                             only merge; other values are rejected)          */
  float sm_scale;         /* softmax scale; <= 0 selects 1/sqrt(D)           */
  int flags;              /* bitwise OR of sv_attn_flags, 0 for none         */

  /* tensors */
  const void* q;          /* bf16 [T, Hq, D]                                 */
  const void* tree_k;     /* bf16 [T, Hkv, D]  K of the tree nodes           */
  const void* tree_v;     /* bf16 [T, Hkv, D]  V of the tree nodes           */
  const void* k_cache;    /* bf16 [num_pages, Hkv, page_size, D]             */
  const void* v_cache;    /* bf16 [num_pages, Hkv, page_size, D]             */
  const int* block_table; /* int32 [B, max_pages_per_seq] logical->physical  */
  const int* ctx_lens;    /* int32 [B] L_b >= 0                              */
  const int* cu_nodes;    /* int32 [B+1] prefix sums of N_b, cu_nodes[0] = 0 */
  const int* parents;     /* int32 [T] sequence-local parent, -1 at node 0,
                             parent[i] < i otherwise                         */
  const int* kv_pages;    /* optional int32 [sum] logical page ids per
                             sequence, ascending and unique, each page <
                             ceil(L_b / page_size); NULL = full verification */
  const int* cu_kv_pages; /* int32 [B+1] prefix sums into kv_pages           */
  void* out;              /* bf16 [T, Hq, D] (written)                       */
  float* lse;             /* optional fp32 [T, Hq]: natural log of the
                             softmax denominator (written if non-NULL)       */
  void* workspace;        /* device scratch, see workspace_size              */
  size_t workspace_bytes;
} sv_attn_params;

/* Bytes of workspace sv_tree_attention needs for these parameters (queries
 * the current device's SM count when num_splits == 0). */
sv_status sv_tree_attention_workspace_size(const sv_attn_params* params, size_t* bytes);

/* The launch plan sv_tree_attention would use for these parameters: the
 * number of KV splits, how they merge (0 = single split, 2 = through
 * workspace partials and the combine kernel) and, if kernel is non-NULL,
 * the kernel (0 = paired, 1 = wide, 2 = dealt; see sv_attn_flags).  For the
 * dealt kernel num_splits is 1 and split_reduce 0: its own combine merges the
 * units that its ranges cut. */
sv_status sv_tree_attention_plan(const sv_attn_params* params, int* num_splits, int* split_reduce, int* kernel);

/* Launches the attention (and, with more than one split, the split combine)
 * on `stream`: one CTA per (KV split, KV head x 128-row tile, sequence) for
 * the paired kernel or per (KV split, KV head x 256-row group, sequence) for
 * the wide one (sv_attn_flags); in batches of 2..64 sequences the longest
 * (context length, or listed pages) are dispatched first.  Hkv x
 * (ceil(max_nodes x G / 128) + 1) must not exceed 65535 (SV_ERR_UNSUPPORTED
 * otherwise). */
sv_status sv_tree_attention(const sv_attn_params* params, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * Greedy acceptance (temperature 0).
 *
 * Defined by: SpecBlock Appendix A.5 (the longest accepted prefix is
 * committed); greedy decoding at T = 0 (SpecBlock section 4, SpecPV
 * Appendix D); the reported accept length excludes the bonus token
 * ("Dynamic Speculative Decoding", Implementation Details: the scheduler
 * keeps accept_length + 1 tokens per request).
 *
 * am[n] = argmax_v logits[n, v], lowest v on ties (-0.0 == +0.0).  Non-root
 * node c is accepted iff tokens[c] == am[parent c] and its parent is
 * accepted (the root always is).  The result per sequence is the deepest
 * accepted node, ties broken by the lexicographically smallest root path of
 * node indices:
 *   accept_len[b]                 its depth (root and bonus excluded)
 *   accepted_nodes[b, 0..a]       its root path (local ids, [0] = 0), the
 *                                 remaining entries up to max_depth are -1
 *   bonus_token[b]                am[last node of the path]
 *   argmax_out[n]                 am[n] for every node (optional)
 *
 * logits: fp32 [T, vocab], rows contiguous.  tokens/parents: int32 [T]
 * (tokens[root] unused).  max_nodes (host) <= 128.  max_depth (host) is the
 * row stride - 1 of accepted_nodes and must be >= every tree's depth.
 * total_nodes <= 65535 (one grid row per node); a larger call returns
 * SV_ERR_UNSUPPORTED.  A sequence whose tree (from the device cu_nodes) has
 * no node or more than 128 is not walked: it gets accept_len 0, bonus_token
 * -1 and a path of -1, and the error word records SV_DEVERR_BAD_TREE; the
 * workspace stays ready for the next call.
 * ---------------------------------------------------------------------- */
sv_status sv_greedy_accept_workspace_size(int batch, int total_nodes, size_t* bytes);

sv_status sv_greedy_accept(const float* logits, int vocab, const int* tokens,
                           const int* parents, const int* cu_nodes, int batch,
                           int total_nodes, int max_nodes, int max_depth,
                           int* argmax_out, int* accept_len, int* accepted_nodes,
                           int* bonus_token, void* workspace, size_t workspace_bytes,
                           sv_stream_t stream);

/* Greedy acceptance that allocates nothing and takes no workspace.
 *
 * No counterpart in the method's description: this is a convenience for
 * callers that cannot allocate device memory when they verify a tree (an
 * engine that gave all free memory to its KV pool at start-up, a plugin whose
 * host framework exposes no allocator, a decode loop that forbids allocation
 * after warm-up).  Same arguments and results as sv_greedy_accept, without
 * the workspace; the scratch it needs lives in a fixed array inside this
 * library's device code, which every GPU that loads the library holds until
 * the process exits.
 *   - Limits: batch <= 1024 and total_nodes <= 8192; larger calls return
 *     SV_ERR_UNSUPPORTED without launching anything.
 *   - The first call on each device looks up that array's device address (a
 *     host-side driver query, with the device current).  With CUDA's lazy
 *     module loading (the default) that first lookup also loads this
 *     library's device code onto the device, which takes device memory once;
 *     so make the first call during warm-up, before any stream capture and
 *     before the point after which the caller may not allocate.  The address
 *     is looked up again when the device's context changes (after a
 *     cudaDeviceReset), and that call loads the device code again.
 *   - Every call uses the same array and clears the part it needs at its
 *     start, so calls that may overlap on the GPU (different streams, or
 *     different host threads without ordering) race with each other and must
 *     not be issued.
 *   - device_error (optional, device int) receives the call's device error
 *     code (0 if none).
 * It calls no cudaMalloc, cudaFree or other allocating routine. */
sv_status sv_greedy_accept_noalloc(const float* logits, int vocab, const int* tokens,
                                   const int* parents, const int* cu_nodes, int batch,
                                   int total_nodes, int max_nodes, int max_depth,
                                   int* argmax_out, int* accept_len, int* accepted_nodes,
                                   int* bonus_token, int* device_error, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * Stochastic (temperature > 0) acceptance of a verified draft tree.
 *
 * Defined by: speculative sampling (SpecPV section 2, citing Leviathan et
 * al.: the emitted tokens follow the target's own sampling distribution) over
 * a token tree (SpecPV section 2, SpecInfer), at the temperatures SpecBlock
 * section 4 and SpecPV Appendix E evaluate.  The pages give no rule for a
 * tree; this follows SpecInfer's multi-step speculative sampling:
 *   p_u = softmax(logits[u] / temperature); the children c of node u (drawn
 *   from draft_probs[u]) are tried in index order against a residual R that
 *   starts as p_u: c (token x) is accepted when u_accept[c] < min(1, R(x) /
 *   q_u(x)) (q_u(x) = 0 accepts); otherwise R <- max(R - q_u, 0) / its sum
 *   (unchanged when the sum is 0).  From the root the walk follows accepted
 *   children to a node z; accept_len is its depth, accepted_nodes its root
 *   path, and bonus_token the smallest x with R_z(0) + ... + R_z(x) >
 *   u_bonus[z] * sum(R_z), R_z being z's residual after all its children
 *   were rejected (p_z for a leaf).
 *
 *   logits       fp32 [total_nodes, vocab], the target's logits per node
 *   draft_probs  fp32 [total_nodes, vocab], per node the probability vector
 *                its children were drawn from (rows of leaves are read only
 *                if the walk ends there and then not at all)
 *   u_accept     fp32 [total_nodes], uniform in [0, 1): node n's test at its
 *                parent (the root's is unused)
 *   u_bonus      fp32 [total_nodes], uniform in [0, 1): the draw at node n
 *   accepted_child (optional) int32 [total_nodes]: per node the local index
 *                of its accepted child, -1 if none
 *   accept_len, accepted_nodes, bonus_token: as for sv_greedy_accept.
 * vocab >= 8 and <= 2^18 (262144); temperature > 0 and finite;
 * max_nodes <= 128.  A larger vocabulary returns SV_ERR_UNSUPPORTED.
 * The workspace (sv_sample_accept_workspace_size bytes) holds per-node
 * scalars between the two launches; it needs no zeroing between calls.
 * ---------------------------------------------------------------------- */
sv_status sv_sample_accept_workspace_size(int batch, int total_nodes, size_t* bytes);

sv_status sv_sample_accept(const float* logits, const float* draft_probs, int vocab,
                           float temperature, const int* tokens, const int* parents,
                           const int* cu_nodes, int batch, int total_nodes, int max_nodes,
                           int max_depth, const float* u_accept, const float* u_bonus,
                           int* accepted_child, int* accept_len, int* accepted_nodes,
                           int* bonus_token, void* workspace, size_t workspace_bytes,
                           sv_stream_t stream);

/* ------------------------------------------------------------------------
 * KV commit of the accepted path, all layers in one launch.
 *
 * Defined by: SpecBlock Appendix A.5 (commit the accepted prefix before the
 * next iteration) and "Dynamic Speculative Decoding", Implementation Details
 * (the KV cache stays consistent with the committed tokens).
 *
 * For every layer l, sequence b and j = 0..accept_len[b]: cache slot
 * s = ctx_lens[b] + j (page block_table[b, s / page_size], row
 * s % page_size) receives, for every KV head, the K and V of tree node
 * accepted_nodes[b, j] (a bit copy).  new_ctx_lens[b] = ctx_lens[b] +
 * accept_len[b] + 1 if non-NULL (ctx_lens[b] when accept_len[b] > max_depth,
 * which commits nothing for b and records SV_DEVERR_DEPTH); it must not
 * alias ctx_lens.  The caller
 * guarantees pages for slots L_b .. L_b + max_depth.  Nothing else changes.
 * The kernel is launched as a programmatic dependent of whatever kernel
 * precedes it on the stream (sv_greedy_accept and sv_sample_accept let it
 * start at once): it waits for that kernel's completion before reading
 * accept_len and accepted_nodes, so the ordering is the stream's as usual.
 *
 * tree_k/tree_v: bf16 [num_layers][T, Hkv, D], layer stride
 * tree_layer_stride elements.  k_cache/v_cache: bf16
 * [num_layers][num_pages, Hkv, page_size, D], layer stride
 * cache_layer_stride elements.  Both strides are multiples of 8.
 * workspace is optional (NULL, or >= 256 bytes zero-filled once) and only
 * receives the error word.  head_dim is a multiple of 8; max_depth + 1,
 * batch and num_layers are each <= 65535 (SV_ERR_UNSUPPORTED otherwise).
 * ---------------------------------------------------------------------- */
sv_status sv_kv_commit(const void* tree_k, const void* tree_v, long long tree_layer_stride,
                       void* k_cache, void* v_cache, long long cache_layer_stride,
                       int num_layers, int num_pages, const int* block_table,
                       int max_pages_per_seq, const int* ctx_lens, const int* cu_nodes,
                       const int* accepted_nodes, const int* accept_len, int batch,
                       int max_depth, int num_kv_heads, int head_dim, int page_size,
                       int* new_ctx_lens, void* workspace, size_t workspace_bytes,
                       sv_stream_t stream);

/* ------------------------------------------------------------------------
 * SpecPV block retrieval: the partial page list of sv_tree_attention.
 *
 * Defined by: SpecPV section 3.2 (the partial KV cache keeps sink blocks,
 * query-dependent retrieved blocks and a local window, attended as one
 * segment; every block's keys are summarised by their element-wise maximum
 * and minimum; blocks are scored against the candidate tokens' query states
 * and the per-query scores reduced by max, mean or last), Appendix C (mean
 * works best) and Appendix D (16-token blocks).
 *
 * A block is one 16-token page.  The score of page p for query q (query
 * head h, KV head h / G) is the largest q . k for a key between the page's
 * minimum and maximum key, sum_d max(q_d kmax_d, q_d kmin_d).  A page's
 * importance is the mean of its scores over every tree node and query head
 * of the sequence (SV_REDUCE_MEAN), their maximum (SV_REDUCE_MAX), or the
 * mean over query heads for the last node in index order (SV_REDUCE_LAST).
 * Sink pages are the first ceil(sink_tokens / 16); window pages hold the
 * last window_tokens tokens; of the pages in between the topk most important
 * are retrieved (equal importance: lower page first).  The list of a
 * sequence is its sink, retrieved and window pages, ascending: exactly the
 * kv_pages / cu_kv_pages input of sv_tree_attention (max_kv_pages <=
 * ceil(sink/16) + topk + ceil(window/16) + 1).
 * ---------------------------------------------------------------------- */

/* Page summaries: for every page of every sequence from logical page
 * first_page[b] on (first_page NULL: all), the element-wise maximum and
 * minimum of the page's valid keys (tokens below ctx_lens[b]), per KV head.
 * After sv_kv_commit, passing first_page = old ctx_lens / 16 and the new
 * lengths refreshes exactly the pages the commit touched.
 *   k_cache     bf16 [num_pages, Hkv, page_size, D] (one layer)
 *   summaries   bf16 [num_pages, Hkv, 2, D]: [.., 0, :] maximum, [.., 1, :]
 *               minimum; pages no sequence uses are left untouched
 *   max_ctx_pages (host) >= every ceil(ctx_lens[b] / 16) - first_page[b]
 *   workspace   optional (NULL, or >= 256 bytes zero-filled once): error word */
sv_status sv_kv_page_summaries(const void* k_cache, int num_pages, int num_kv_heads, int head_dim, int page_size,
                               const int* block_table, int max_pages_per_seq, const int* ctx_lens,
                               const int* first_page, int batch, int max_ctx_pages, void* summaries,
                               void* workspace, size_t workspace_bytes, sv_stream_t stream);

typedef enum sv_reduce { SV_REDUCE_MEAN = 0, SV_REDUCE_MAX = 1, SV_REDUCE_LAST = 2 } sv_reduce;

typedef struct sv_retrieve_params {
  int batch;              /* B                                              */
  int num_q_heads;        /* Hq                                             */
  int num_kv_heads;       /* Hkv                                            */
  int head_dim;           /* D: 64 or 128                                   */
  int page_size;          /* 16                                             */
  int num_pages;          /* pages in the pool                              */
  int total_nodes;        /* T = cu_nodes[B]                                */
  int max_pages_per_seq;  /* row length of block_table                      */
  int max_ctx_pages;      /* host: max_b ceil(ctx_lens[b] / 16), <= 16384   */
  int sink_tokens;
  int window_tokens;
  int topk;               /* pages retrieved between sink and window        */
  int reduce;             /* sv_reduce                                      */
  const void* q;          /* bf16 [T, Hq, D] the tree nodes' queries        */
  const void* summaries;  /* bf16 [num_pages, Hkv, 2, D] (sv_kv_page_summaries) */
  const int* block_table; /* int32 [B, max_pages_per_seq]                   */
  const int* ctx_lens;    /* int32 [B]                                      */
  const int* cu_nodes;    /* int32 [B+1]                                    */
  int* kv_pages;          /* out: int32, the lists packed in sequence order */
  int* cu_kv_pages;       /* out: int32 [B+1] prefix sums                   */
  float* scores;          /* optional out: fp32 [B, max_ctx_pages], the
                             importance of every candidate page, -inf for
                             the others                                     */
  size_t kv_pages_capacity; /* entries of kv_pages (>= B x the list bound)  */
  void* workspace;        /* sv_retrieve_pages_workspace_size bytes         */
  size_t workspace_bytes;
} sv_retrieve_params;

sv_status sv_retrieve_pages_workspace_size(int batch, int num_kv_heads, int head_dim, int max_ctx_pages,
                                           size_t* bytes);

sv_status sv_retrieve_pages(const sv_retrieve_params* params, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * SpecPV full / partial verification schedule.
 *
 * Defined by: SpecPV section 3.3 (partial verification begins after a full
 * verification initialises the partial cache; the tokens accepted under
 * partial verification sit in a buffer, and exceeding its limit triggers a
 * full verification that refreshes the cache; before a full verification the
 * partially verified tokens are prepended to the new candidates) and
 * Appendix C (the limit is one verification step's tokens plus 20).
 *
 * Host bookkeeping per sequence.  A partial step attends the refresh's page
 * list plus the pages the buffer has grown into (sv_partial_list_extend).  A
 * full step re-verifies the buffer: its tree is the buffered tokens as a
 * chain ahead of the new candidates, over the context as it was at the
 * refresh (ctx_lens = refresh_ctx_len), attended in full; its commit
 * rewrites the buffered slots with their exact K/V, then the summaries of
 * the touched pages and the retrieval are refreshed.
 * ---------------------------------------------------------------------- */
typedef enum sv_verify_kind { SV_VERIFY_PARTIAL = 0, SV_VERIFY_FULL = 1 } sv_verify_kind;

typedef struct sv_specpv_seq {
  int has_partial_cache;  /* a full verification has built the partial cache */
  int refresh_ctx_len;    /* committed length at that full verification        */
  int buffer_tokens;      /* tokens committed by partial steps since            */
} sv_specpv_seq;

/* The verification the next step of a sequence needs, given the tokens that
 * step can commit at most (the tree's depth + 1) and the buffer limit. */
sv_verify_kind sv_specpv_next(const sv_specpv_seq* seq, int step_tokens, int buffer_limit);

/* Updates the bookkeeping after a step of the given kind committed, leaving
 * ctx_len_after committed tokens. */
sv_status sv_specpv_after(sv_specpv_seq* seq, sv_verify_kind kind, int ctx_len_after);

/* Partial lists between refreshes: sequence b's list made at the refresh
 * (ref_pages[ref_cu[b] .. ref_cu[b+1]), for context length ref_ctx_lens[b])
 * plus the logical pages ceil(ref_ctx_lens[b] / 16) .. ceil(ctx_lens[b] / 16)
 * - 1 that the buffer has grown into; written packed, in sequence order, with
 * prefix sums in cu_kv_pages [B+1].  kv_pages needs room for the refresh
 * lists plus the new pages.  workspace optional (error word). */
sv_status sv_partial_list_extend(const int* ref_pages, const int* ref_cu, const int* ref_ctx_lens,
                                 const int* ctx_lens, int batch, int* kv_pages, int* cu_kv_pages,
                                 void* workspace, size_t workspace_bytes, sv_stream_t stream);

/* The trees of a full verification that follows partial ones (SpecPV
 * section 3.3: before a full verification, the partially verified tokens are
 * prepended to the new candidates; the full KV cache is used).
 *
 * Per sequence b: the buffered tokens buffer_tokens[buffer_cu[b] ..
 * buffer_cu[b+1]) (the nb tokens committed since the last full
 * verification, positions R .. L-1 with R = refresh_ctx_len) and the
 * candidate tree (cand_parents / cand_tokens [cand_cu[b] .. cand_cu[b+1]),
 * local ids, root = the last accepted token at position L).  Output, packed
 * in sequence order with prefix sums cu_nodes [B+1]: node j < nb is buffered
 * token j with parent j - 1 (the chain's first node is the root), node
 * nb + i is candidate node i with parent nb + cand_parents[i], and the
 * candidate root's parent is nb - 1 (-1 when nb = 0: the candidate tree
 * unchanged).
 *
 * The full step then runs sv_tree_attention, sv_greedy_accept and
 * sv_kv_commit on these trees with ctx_lens = R (full KV): every buffered
 * token is checked again like a candidate (node j is accepted when its token
 * is the target's arg-max after node j - 1; a rejection ends the path there
 * and the bonus token replaces the buffered one), and the commit writes slots
 * R .. R + a, rewriting the buffered slots with this forward's K/V.  The
 * caller's host sizes: total_nodes = total candidate nodes + sum nb;
 * max_nodes = max(nb + candidate nodes) <= 128; max_depth = max(nb +
 * candidate depth).  Device errors: a sequence with nb < 0, no candidate
 * node or more than 128 combined nodes -> SV_DEVERR_BAD_TREE; a candidate
 * parent not before its child -> SV_DEVERR_BAD_PARENT (the tree is still
 * written).  parents/tokens need room for all combined nodes; buffer_tokens
 * may be NULL when every buffer is empty; workspace optional (error word). */
sv_status sv_specpv_full_trees(const int* cand_parents, const int* cand_tokens, const int* cand_cu,
                               const int* buffer_tokens, const int* buffer_cu, int batch,
                               int* parents, int* tokens, int* cu_nodes, void* workspace,
                               size_t workspace_bytes, sv_stream_t stream);

/* Diagnostics: per-CTA phase tracing of sv_tree_attention.
 *
 * After this call, every sv_tree_attention launch (until the buffer is
 * replaced, or removed with buffer = NULL) writes, for each of its CTAs in
 * linear grid order, kSvTraceSlots 64-bit words: [0] %globaltimer (ns) at
 * CTA start, [1..] SM clock cycles since CTA start at the phase boundaries
 * listed in sv_trace_event.  A CTA beyond the buffer records nothing.  The
 * setting is process-wide and not synchronised with launches in flight; use
 * it from one thread while no launch is being recorded into a stream. */
enum { kSvTraceSlots = 16 };
typedef enum sv_trace_event {
  SV_TRACE_START_NS = 0,      /* globaltimer at CTA start                      */
  SV_TRACE_PROLOGUE = 1,      /* barriers, TMEM and descriptor prefetch done   */
  SV_TRACE_INPUTS = 2,        /* after the wait on the preceding grid          */
  SV_TRACE_FIRST_IDS = 3,     /* producer: first page ids read                 */
  SV_TRACE_FIRST_MMA = 4,     /* MMA issuer: Q and the first K tile landed     */
  SV_TRACE_FIRST_S = 5,       /* softmax (row tile 0): first scores ready      */
  SV_TRACE_LOOP_END = 6,      /* softmax (row tile 0): last P handed over      */
  SV_TRACE_O_READY = 7,       /* softmax (row tile 0): final O complete        */
  SV_TRACE_EPILOGUE = 8,      /* output or partial written / parked            */
  SV_TRACE_MERGE_READY = 9,   /* reserved (no current kernel records it)       */
  SV_TRACE_MERGE_DONE = 10,   /* reserved (no current kernel records it)       */
  SV_TRACE_EXIT = 11,         /* before TMEM release                           */
  SV_TRACE_TREE_MASK = 12     /* softmax (row tile 0): ancestor masks built    */
} sv_trace_event;

sv_status sv_set_trace_buffer(void* buffer, size_t bytes);

/* Reads the error word of a workspace (waits for `stream`), stores it in
 * *code (host) and resets it to zero.  Returns SV_ERR_TIMEOUT if it held
 * SV_DEVERR_TIMEOUT, SV_ERR_DEVICE for any other nonzero code, SV_OK
 * otherwise. */
sv_status sv_get_device_error(void* workspace, int* code, sv_stream_t stream);

/* Diagnostics: exercises the bounded wait every kernel of this library uses
 * on its mbarriers.  Launches one CTA that waits for a barrier nothing will
 * complete.  With abort_after_ns == 0 the wait gives up after the library's
 * limit (2 s); with 0 < abort_after_ns < 2e9 another warp of the CTA raises
 * the abort flag after that long, as a failing role of a kernel does.  Either
 * way the kernel records SV_DEVERR_TIMEOUT in the error word of `workspace`
 * (a device int, zero before the call) and returns; the context stays
 * usable.  Read the outcome with sv_get_device_error. */
sv_status sv_selftest_bounded_wait(void* workspace, long long abort_after_ns, sv_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* SV_H_ */
