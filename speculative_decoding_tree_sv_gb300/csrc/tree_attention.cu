// Tree-verification attention for sm_103a.
//
// What it computes (SpecBlock Appendix A.5: every drafted node is scored in
// one target forward; Appendix A.2: a node sees the verified prefix and its
// on-path ancestors; SpecPV section 3.2: a partial cache of retained blocks is
// attended as one continuous KV segment): for every tree node i and query
// head h,  out[i,h] = softmax(scale * q[i,h] K^T + mask) V  over the context
// keys followed by the tree keys, where the tree part of the mask keeps only
// ancestors-or-self of i.
//
// Design (one CTA per (KV split, KV head x 256-row group, sequence)):
//   * The M dimension of the contraction is (tree node x query head of the
//     GQA group): rows r = node * G + g, two 128-row tiles per CTA.
//   * Context K/V pages (16 tokens, head-major inside a page) are gathered
//     with TMA, eight pages (128 keys) per tile, 128-byte swizzled, into a
//     ring of smem stages.  The tree's own K/V form one extra tile.
//   * tcgen05.mma computes S = Q K^T (both operands K-major in smem) into
//     TMEM; softmax warps read S with tcgen05.ld (one row per thread), apply
//     the mask and an online, lazily rescaled softmax in base 2 (packed
//     two-lane fp32 arithmetic), write P as bf16 back into the S columns, and
//     tcgen05.mma accumulates O += P V (P from TMEM, V MN-major in smem).
//   * Warp roles: warp 0 loads (TMA), warp 1 issues MMAs (one thread),
//     warps 4-7 and 8-11 run the softmax of row tiles 0 and 1.  The MMA
//     issue order S0 S1 | PV0 S0' | PV1 S1' ... keeps the tensor core busy
//     while the two softmax groups alternate.
//   * KV splits are merged one of two ways.  Inside a cluster: the splits of
//     one (sequence, head group) form a thread-block cluster, so they are
//     co-resident; each writes its partial (O / l, log2-sum-exp) to the
//     workspace, signals its peers' mbarriers, waits for theirs (bounded)
//     and merges a slice of the rows from L2.  With a second kernel: for
//     very long contexts, where more splits than fit in co-resident clusters
//     pay off, the splits write partials that a combine kernel merges.
//   * Launches allow programmatic dependent launch: the prologue (barriers,
//     TMEM, descriptor prefetch) runs before the wait on the previous grid.
#include <math.h>

#include <mutex>

#include "sv_device.cuh"

namespace sv {
namespace attn {

constexpr int kThreads = 384;
// Registers per thread after the split: 128 x 56 (load + MMA group) + 256 x
// 224 (softmax groups) = 64512 = 384 x 168, the launch allocation.
constexpr int kRegsControl = 56;
constexpr int kRegsSoftmax = 224;
constexpr int kBlockN = 128;       // keys per tile (8 pages)
constexpr int kTileRows = 128;     // rows per M tile
constexpr int kCtaRows = 256;      // two M tiles per CTA
constexpr int kPagesPerTile = kBlockN / 16;
constexpr int kMaxClusterSplits = 16;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: defer O rescale until max grows by 2^8
constexpr float kLn2 = 0.69314718055994530942f;

enum ReduceMode : int { kReduceNone = 0, kReduceCluster = 1, kReduceGlobal = 2 };

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;                   // 128-byte column halves
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr uint32_t kHalfBytes = 128u * 128u;      // 128 rows x 128 B
  static constexpr uint32_t kQTileBytes = kTileRows * D * 2;
  static constexpr uint32_t kKVTileBytes = kBlockN * D * 2;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + 2 * kQTileBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kKVTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kStages * kKVTileBytes;
  static constexpr uint32_t kBarBytes = 512;
  static constexpr uint32_t kSmemBytes = kOffBar + kBarBytes + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128;
  static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
  // epilogue staging of output rows (one padded row per softmax thread),
  // over the Q/K/V stages once every MMA is done
  static constexpr uint32_t kStageStride = D * 4 + 16;
  static constexpr uint32_t kOffStage = 0;
  static_assert(kOffStage + 2 * kTileRows * kStageStride <= kOffBar, "staging must fit below the barriers");
};

struct Params {
  const int* block_table;
  const int* ctx_lens;
  const int* cu_nodes;
  const int* parents;
  const int* kv_pages;
  const int* cu_kv_pages;
  __nv_bfloat16* out;
  float* lse;
  __nv_bfloat16* part_o;  // split partials O / l (bf16), [splits][T * Hq][D]
  float* part_lse;        // split partials log2-sum-exp, [splits][T * Hq]
  int* err;
  unsigned long long* trace;  // optional per-CTA phase timestamps
  long long trace_ctas;
  int num_q_heads;
  int group;  // G
  int num_pages;
  int max_pages_per_seq;
  int num_splits;
  int reduce_mode;
  int total_nodes;
  int groups_per_seq;
  float scale_log2;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    tree_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                          const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_tk,
                          const __grid_constant__ CUtensorMap tm_tv, const __grid_constant__ Params p) {
  using C = Cfg<D>;
  constexpr int NST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int split = blockIdx.x;
  const int kh = blockIdx.y / p.groups_per_seq;
  const int mg = blockIdx.y % p.groups_per_seq;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const bool cluster_mode = p.reduce_mode == kReduceCluster;
  // phase tracing (diagnostics): no live registers when it is off
  long long* trace_clk0 = reinterpret_cast<long long*>(smem + C::kOffBar + C::kBarBytes - 8);
  auto mark = [&](int ev) {
    if (p.trace != nullptr) {
      const long long id = blockIdx.x + static_cast<long long>(gridDim.x) *
                                            (blockIdx.y + static_cast<long long>(gridDim.y) * blockIdx.z);
      if (id < p.trace_ctas)
        p.trace[id * kSvTraceSlots + ev] = static_cast<unsigned long long>(clock64() - *trace_clk0);
    }
  };
  if (p.trace != nullptr && threadIdx.x == 0) {
    *trace_clk0 = clock64();
    const long long id =
        blockIdx.x + static_cast<long long>(gridDim.x) * (blockIdx.y + static_cast<long long>(gridDim.y) * blockIdx.z);
    if (id < p.trace_ctas) p.trace[id * kSvTraceSlots + SV_TRACE_START_NS] = globaltimer_ns();
  }

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NST;
  uint64_t* k_empty = v_full + NST;
  uint64_t* v_empty = k_empty + NST;
  uint64_t* s_full = v_empty + NST;  // [2]
  uint64_t* p_full = s_full + 2;     // [2]
  uint64_t* o_final = p_full + 2;    // [2]
  uint64_t* drain = o_final + 2;
  uint64_t* published = drain + 1;   // cluster merge: every peer's partial is in the workspace
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(published + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never_set = abort_flag + 1;  // drains wait on copies even after an abort

  // ---- prologue that reads no input: it may overlap the previous grid
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(v_full + i, 1);
      mbar_init(k_empty + i, 1);
      mbar_init(v_empty + i, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full + t, 1);
      mbar_init(p_full + t, kTileRows);
      mbar_init(o_final + t, 1);
    }
    mbar_init(drain, 1);
    mbar_init(published, p.num_splits);
    *abort_flag = 0;
    *never_set = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kc);
    tma_prefetch_desc(&tm_vc);
    tma_prefetch_desc(&tm_tk);
    tma_prefetch_desc(&tm_tv);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every CTA of a cluster reaches this point: peers' barriers are initialised
  // before anyone can arrive on them remotely
  if (cluster_mode) cluster_sync_all();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) mark(SV_TRACE_PROLOGUE);
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x == 0) mark(SV_TRACE_INPUTS);

  const int n0 = p.cu_nodes[b];
  const int N = p.cu_nodes[b + 1] - n0;
  const int L = p.ctx_lens[b];
  const int rows_total = N * G;
  const int row0 = mg * kCtaRows;
  // uniform over the cluster (its CTAs differ only in the split)
  if (row0 < rows_total) {
  const bool tile1 = row0 + kTileRows < rows_total;
  const bool partial = p.kv_pages != nullptr;
  int n_pages, kvp0 = 0;
  if (partial) {
    kvp0 = p.cu_kv_pages[b];
    n_pages = p.cu_kv_pages[b + 1] - kvp0;
  } else {
    n_pages = (L + 15) >> 4;
  }
  // Only the last listed page can hold fewer than 16 context tokens.
  int last_page_tokens = 16;
  if (n_pages > 0) {
    const int lp = partial ? p.kv_pages[kvp0 + n_pages - 1] : n_pages - 1;
    last_page_tokens = min(16, max(0, L - 16 * lp));
  }
  const int t_ctx = (n_pages + kPagesPerTile - 1) / kPagesPerTile;
  const int t_all = t_ctx + 1;  // + the tree tile
  const int jb = static_cast<int>(static_cast<long long>(split) * t_all / p.num_splits);
  const int je = static_cast<int>(static_cast<long long>(split + 1) * t_all / p.num_splits);
  const int ntiles = je - jb;
  const bool work = ntiles > 0;

  if (!work && p.reduce_mode == kReduceGlobal) {
    // empty split: publish an empty partial for our rows
    if (threadIdx.x < kCtaRows) {
      const int row = row0 + threadIdx.x;
      if (row < rows_total) {
        const int node = row / G, g = row - (row / G) * G;
        p.part_lse[(static_cast<size_t>(split) * p.total_nodes + n0 + node) * p.num_q_heads + kh * G + g] =
            -INFINITY;
      }
    }
  } else if (warp < 4) {
    regs_decrease<kRegsControl>();
    if (work && warp == 0) {
      // ------------------------------------------------------------ producer
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, (tile1 ? 2u : 1u) * C::kQTileBytes);
        for (int t = 0; t < (tile1 ? 2 : 1); ++t)
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_3d(smem + C::kOffQ + t * C::kQTileBytes + h * C::kHalfBytes, &tm_q, q_full, h * 64, kh * G,
                        n0 + (row0 + t * kTileRows) / G);
      }
      for (int it = 0; it < ntiles; ++it) {
        const int j = jb + it;
        const int st = it % NST;
        const uint32_t ph = (it / NST) & 1;
        const bool ctx = j < t_ctx;
        int phys = 0;
        if (ctx && lane < kPagesPerTile) {
          const int ps = min(j * kPagesPerTile + lane, n_pages - 1);  // ragged tail repeats the last page
          int lp = partial ? p.kv_pages[kvp0 + ps] : ps;
          if (lp < 0 || lp >= p.max_pages_per_seq) {
            report_error(p.err, SV_DEVERR_BAD_PAGE);
            lp = 0;
          }
          phys = p.block_table[static_cast<size_t>(b) * p.max_pages_per_seq + lp];
          if (phys < 0 || phys >= p.num_pages) {
            report_error(p.err, SV_DEVERR_BAD_PAGE);
            phys = 0;
          }
        }
        // K tile
        if (it >= NST) {
          int w = (lane == 0) ? (mbar_wait(k_empty + st, ph ^ 1u, abort_flag) ? 1 : 0) : 0;
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
        }
        if (lane == 0) mbar_arrive_expect_tx(k_full + st, C::kKVTileBytes);
        __syncwarp();
        uint8_t* kdst = smem + C::kOffK + st * C::kKVTileBytes;
        if (ctx) {
          if (lane < kPagesPerTile)
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_4d(kdst + h * C::kHalfBytes + lane * 2048, &tm_kc, k_full + st, h * 64, 0, kh, phys);
        } else if (lane == 0) {
          for (int h = 0; h < C::kHalves; ++h) tma_load_3d(kdst + h * C::kHalfBytes, &tm_tk, k_full + st, h * 64, kh, n0);
        }
        k_issued = it + 1;
        // V tile
        if (it >= NST) {
          int w = (lane == 0) ? (mbar_wait(v_empty + st, ph ^ 1u, abort_flag) ? 1 : 0) : 0;
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
        }
        if (lane == 0) mbar_arrive_expect_tx(v_full + st, C::kKVTileBytes);
        __syncwarp();
        uint8_t* vdst = smem + C::kOffV + st * C::kKVTileBytes;
        if (ctx) {
          if (lane < kPagesPerTile)
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_4d(vdst + h * C::kHalfBytes + lane * 2048, &tm_vc, v_full + st, h * 64, 0, kh, phys);
        } else if (lane == 0) {
          for (int h = 0; h < C::kHalves; ++h) tma_load_3d(vdst + h * C::kHalfBytes, &tm_tv, v_full + st, h * 64, kh, n0);
        }
        v_issued = it + 1;
      }
      if (!ok && lane == 0) {
        // Timed out: stop the other roles, then let our copies land before exit.
        report_error(p.err, SV_DEVERR_TIMEOUT);
        *abort_flag = 1;
        mbar_wait(q_full, 0, never_set);
        for (int it = max(0, k_issued - NST); it < k_issued; ++it)
          mbar_wait(k_full + (it % NST), (it / NST) & 1, never_set);
        for (int it = max(0, v_issued - NST); it < v_issued; ++it)
          mbar_wait(v_full + (it % NST), (it / NST) & 1, never_set);
      }
    } else if (work && warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kBlockN, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
        const int nt = tile1 ? 2 : 1;
        const uint32_t q_base = smem_u32(smem + C::kOffQ);
        const uint32_t k_base = smem_u32(smem + C::kOffK);
        const uint32_t v_base = smem_u32(smem + C::kOffV);
        bool ok = mbar_wait(q_full, 0, abort_flag);
        auto issue_qk = [&](int t, int st) {
          const uint32_t d = tmem + (t ? C::kColS1 : C::kColS0);
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
            const uint64_t a = smem_desc_sw128(q_base + t * C::kQTileBytes + off, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(k_base + st * C::kKVTileBytes + off, 16, 1024);
            umma_ss(d, a, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
          }
        };
        auto issue_pv = [&](int t, int st, bool accumulate) {
          const uint32_t d = tmem + (t ? C::kColO1 : C::kColO0);
          const uint32_t a = tmem + (t ? C::kColS1 : C::kColS0);
  #pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk) {
            const uint64_t bdesc = smem_desc_sw128(v_base + st * C::kKVTileBytes + kk * 2048, C::kHalfBytes, 1024);
            umma_ts(d, a + kk * 8, bdesc, idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
          }
        };
        if (ok) ok = mbar_wait(k_full, 0, abort_flag);
        if (ok) {
          tc_fence_after();
          mark(SV_TRACE_FIRST_MMA);
          for (int t = 0; t < nt; ++t) {
            issue_qk(t, 0);
            umma_commit(s_full + t);
          }
          umma_commit(k_empty);
        }
        for (int it = 0; ok && it < ntiles; ++it) {
          const int st = it % NST;
          const uint32_t ph = (it / NST) & 1;
          const int nx = it + 1;
          const int st2 = nx % NST;
          const uint32_t ph2 = (nx / NST) & 1;
          if (!mbar_wait(v_full + st, ph, abort_flag)) { ok = false; break; }
          for (int t = 0; t < nt; ++t) {
            if (!mbar_wait(p_full + t, it & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            issue_pv(t, st, it > 0);
            if (nx < ntiles) {
              if (t == 0) {
                if (!mbar_wait(k_full + st2, ph2, abort_flag)) { ok = false; break; }
                tc_fence_after();
              }
              issue_qk(t, st2);
              umma_commit(s_full + t);
            }
          }
          if (!ok) break;
          umma_commit(v_empty + st);
          if (nx < ntiles) umma_commit(k_empty + st2);
        }
        if (ok) {
          for (int t = 0; t < nt; ++t) umma_commit(o_final + t);
        } else {
          report_error(p.err, SV_DEVERR_TIMEOUT);
          *abort_flag = 1;
          umma_commit(drain);  // let issued MMAs finish before TMEM is freed
          mbar_wait(drain, 0, never_set);
        }
      }
      __syncwarp();
    }
  } else {
    regs_increase<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int qw = warp & 3;
    const int r = qw * 32 + lane;
    const int r_cta = t * kTileRows + r;
    const int row = row0 + r_cta;
    const bool row_exists = row < rows_total;
    const bool active = work && (t == 0 || tile1);  // warp-uniform
    const int node = row / G;
    const int g = row - node * G;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    const uint32_t col_s = t ? C::kColS1 : C::kColS0;
    const uint32_t col_o = t ? C::kColO1 : C::kColO0;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    if (active) {
        // ancestor-or-self bitmask of this row's node (only the split that
        // owns the tree tile needs it)
        uint32_t anc0 = 0, anc1 = 0, anc2 = 0, anc3 = 0;
        if (je == t_all && row_exists) {
          int c = node;
          for (int step = 0; step < kMaxNodes && c >= 0 && c < kMaxNodes; ++step) {
            const uint32_t bit = 1u << (c & 31);
            if ((c >> 5) == 0) anc0 |= bit;
            else if ((c >> 5) == 1) anc1 |= bit;
            else if ((c >> 5) == 2) anc2 |= bit;
            else anc3 |= bit;
            if (c == 0) break;
            const int pc = p.parents[n0 + c];
            if (pc < 0 || pc >= c) {
              report_error(p.err, SV_DEVERR_BAD_PARENT);
              break;
            }
            c = pc;
          }
        }

        if (t == 0 && r == 0 && je == t_all) mark(SV_TRACE_TREE_MASK);
        for (int it = 0; it < ntiles; ++it) {
          const int j = jb + it;
          // warp-uniform outcome: the TMEM loads below are warp-collective
          if (!__all_sync(0xffffffffu, mbar_wait(s_full + t, it & 1, abort_flag))) { ok = false; break; }
          tc_fence_after();
          if (it == 0 && t == 0 && r == 0) mark(SV_TRACE_FIRST_S);
          uint32_t sr[kBlockN];
  #pragma unroll
          for (int c = 0; c < kBlockN / 32; ++c)
            tmem_ld32(lane_base + col_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + c * 32));
          tmem_ld_wait();
          // mask: only the ragged last context tile and the tree tile need one
          constexpr uint32_t kNegInf = 0xFF800000u;
          if (j >= t_ctx) {
  #pragma unroll
            for (int k = 0; k < kBlockN; ++k) {
              const uint32_t w = (k < 32) ? anc0 : (k < 64) ? anc1 : (k < 96) ? anc2 : anc3;
              if (!((k < N) && ((w >> (k & 31)) & 1u))) sr[k] = kNegInf;
            }
          } else if (j == t_ctx - 1) {
            const int nvalid = (n_pages - kPagesPerTile * j - 1) * 16 + last_page_tokens;
  #pragma unroll
            for (int k = 0; k < kBlockN; ++k)
              if (k >= nvalid) sr[k] = kNegInf;
          }
          // row maximum of the raw scores (scale > 0 commutes with max)
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
  #pragma unroll
          for (int k = 0; k < kBlockN; k += 8) {
            mx0 = max3(mx0, __uint_as_float(sr[k + 0]), __uint_as_float(sr[k + 1]));
            mx1 = max3(mx1, __uint_as_float(sr[k + 2]), __uint_as_float(sr[k + 3]));
            mx2 = max3(mx2, __uint_as_float(sr[k + 4]), __uint_as_float(sr[k + 5]));
            mx3 = max3(mx3, __uint_as_float(sr[k + 6]), __uint_as_float(sr[k + 7]));
          }
          const float tmax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * p.scale_log2;
          const float m_new = fmaxf(m_run, tmax);
          const bool grow = m_new > m_run + kRescaleThreshold;
          // The O rescale reads and writes TMEM with warp-collective
          // instructions: the whole warp takes it when any row needs it
          // (rows that do not are scaled by 1).
          if (it > 0 && __any_sync(0xffffffffu, grow)) {
            // O already holds earlier tiles (their PV finished before this S
            // was committed): rescale it and the running sum.
            {
              const float f = grow ? ex2(m_run - m_new) : 1.f;
              l_run *= f;
              const uint64_t f2 = f2_pack(f, f);
              uint32_t o[32];
  #pragma unroll
              for (int c = 0; c < D / 32; ++c) {
                tmem_ld32(lane_base + col_o + c * 32, o);
                tmem_ld_wait();
  #pragma unroll
                for (int k = 0; k < 32; k += 2) {
                  const uint64_t v = f2_mul(f2_pack(__uint_as_float(o[k]), __uint_as_float(o[k + 1])), f2);
                  o[k] = static_cast<uint32_t>(v);
                  o[k + 1] = static_cast<uint32_t>(v >> 32);
                }
                tmem_st32(lane_base + col_o + c * 32, o);
              }
              tmem_st_wait();
            }
          }
          if (grow) m_run = m_new;
          const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
          // p = 2^(s * scale_log2 - m), packed two at a time
          const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
          const uint64_t nm2 = f2_pack(-m_use, -m_use);
          uint64_t acc0 = 0, acc1 = 0;
          uint32_t pk[kBlockN / 2];
  #pragma unroll
          for (int k = 0; k < kBlockN; k += 4) {
            const uint64_t a = f2_fma(f2_pack(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), sc2, nm2);
            const uint64_t b = f2_fma(f2_pack(__uint_as_float(sr[k + 2]), __uint_as_float(sr[k + 3])), sc2, nm2);
            const float p0 = ex2(f2_lo(a)), p1 = ex2(f2_hi(a));
            const float p2 = ex2(f2_lo(b)), p3 = ex2(f2_hi(b));
            acc0 = f2_add(acc0, f2_pack(p0, p1));
            acc1 = f2_add(acc1, f2_pack(p2, p3));
            pk[k >> 1] = pack_bf16x2(p0, p1);
            pk[(k >> 1) + 1] = pack_bf16x2(p2, p3);
          }
          const uint64_t acc = f2_add(acc0, acc1);
          l_run += f2_lo(acc) + f2_hi(acc);
  #pragma unroll
          for (int c = 0; c < kBlockN / 64; ++c)
            tmem_st32(lane_base + col_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(pk + c * 32));
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(p_full + t);
        }
        if (t == 0 && r == 0) mark(SV_TRACE_LOOP_END);

      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_final + t, 0, abort_flag));
      if (t == 0 && r == 0) mark(SV_TRACE_O_READY);
      if (!ok && lane == 0) {
        report_error(p.err, SV_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
    }

    // ---------------------------------------------------------- epilogue
    const bool have_o = active && ok;  // warp-uniform
    if (have_o) tc_fence_after();
    const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
    const float lse2 = (have_o && l_run > 0.f) ? m_run + log2f(l_run) : -INFINITY;
    const size_t orow = static_cast<size_t>(n0 + node) * p.num_q_heads + kh * G + g;
    // Output rows leave through shared memory: each thread parks its row
    // (one TMEM lane) in a padded staging row over the dead Q/K/V stages
    // (every MMA finished before o_final fired), then the warp writes whole
    // rows, lane l moving chunk l, so global stores are coalesced.
    const bool partial_out = p.reduce_mode != kReduceNone;
    if (have_o) {
      uint32_t o[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(lane_base + col_o + c * 32, *reinterpret_cast<uint32_t(*)[32]>(o + c * 32));
      tmem_ld_wait();
      uint8_t* stage = smem + C::kOffStage + (warp - 4) * 32 * C::kStageStride;
      uint8_t* mine = stage + lane * C::kStageStride;
#pragma unroll
      for (int v = 0; v < D / 8; ++v) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l);
        w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l);
        w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l);
        w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l);
        reinterpret_cast<uint4*>(mine)[v] = w;
      }
      __syncwarp();
      // rows of D bf16 = D / 8 16-byte chunks; the warp stores 256 / D rows per
      // instruction
      constexpr int kChunks = D / 8;
      constexpr int kRowsPerPass = 32 / kChunks;
      const int wrow0 = row0 + t * kTileRows + qw * 32;
      const int nrows = min(32, rows_total - wrow0);
      const size_t split_base = partial_out ? static_cast<size_t>(split) * p.total_nodes * p.num_q_heads : 0;
      const long long my_out_row = static_cast<long long>(split_base + orow);  // this lane's row
      __nv_bfloat16* const base = partial_out ? p.part_o : p.out;
      for (int rb = 0; rb < nrows; rb += kRowsPerPass) {
        const int rr = rb + lane / kChunks;
        const long long grow_out = __shfl_sync(0xffffffffu, my_out_row, min(rr, 31));
        if (rr < nrows)
          reinterpret_cast<uint4*>(base + grow_out * D)[lane % kChunks] =
              reinterpret_cast<const uint4*>(stage + rr * C::kStageStride)[lane % kChunks];
      }
    }
    if (p.reduce_mode == kReduceNone) {
      if (have_o && row_exists && p.lse != nullptr) p.lse[orow] = lse2 * kLn2;
      if (r_cta == 0) mark(SV_TRACE_EPILOGUE);
    } else if (p.reduce_mode == kReduceGlobal) {
      if (row_exists && (t == 0 || tile1))
        p.part_lse[static_cast<size_t>(split) * p.total_nodes * p.num_q_heads + orow] = lse2;
    } else {
      // ---- merge inside the cluster (one CTA per split, co-resident)
      // Each CTA has written its partial rows (O / l and log2-sum-exp, fp32)
      // to the workspace; it tells its peers through their mbarriers
      // (release at cluster scope), waits until every peer has done the same
      // (bounded), then merges its own slice of the rows from the peers'
      // partials, which sit in L2.  Global memory outlives the CTAs: no exit
      // handshake is needed.
      const int S = p.num_splits;
      const int rank = static_cast<int>(cluster_ctarank());
      const size_t split_stride = static_cast<size_t>(p.total_nodes) * p.num_q_heads;
      if (row_exists && (t == 0 || tile1)) p.part_lse[static_cast<size_t>(split) * split_stride + orow] = lse2;
      if (r_cta == 0) mark(SV_TRACE_EPILOGUE);
      named_barrier(1, 2 * kTileRows);
      if (threadIdx.x == 4 * 32) {
        for (int rk = 0; rk < S; ++rk) mbar_arrive_cluster(mapa_shared(smem_u32(published), rk));
      }
      if (mbar_wait_cluster(published, 0)) {
        if (r_cta == 0) mark(SV_TRACE_MERGE_READY);
        constexpr int E = D / 32;  // output elements per lane
        constexpr int R = 2;       // rows merged together (their loads overlap)
        const int rows_cta = min(kCtaRows, rows_total - row0);
        const int slice = (rows_cta + S - 1) / S;
        const int lo = rank * slice, hi = min(rows_cta, lo + slice);
        for (int rb = lo + (warp - 4) * R; rb < hi; rb += 8 * R) {
          size_t out_row[R];
          float ls[R];
          float4 v4[R][kMaxClusterSplits];
#pragma unroll
          for (int q = 0; q < R; ++q) {
            const int rr = min(rb + q, hi - 1);  // a duplicate row is merged twice, harmlessly
            const int grow = row0 + rr;
            const int gnode = grow / G;
            out_row[q] = static_cast<size_t>(n0 + gnode) * p.num_q_heads + kh * G + (grow - gnode * G);
            ls[q] = (lane < S) ? __ldcg(p.part_lse + lane * split_stride + out_row[q]) : -INFINITY;
#pragma unroll
            for (int s = 0; s < kMaxClusterSplits; ++s) {
              if (s < S) {
                const __nv_bfloat16* src = p.part_o + (s * split_stride + out_row[q]) * D + lane * E;
                if constexpr (E == 4) {
                  const uint2 v = __ldcg(reinterpret_cast<const uint2*>(src));
                  v4[q][s] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                                         __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
                } else {
                  const uint32_t v = __ldcg(reinterpret_cast<const unsigned int*>(src));
                  v4[q][s] = make_float4(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u), 0.f, 0.f);
                }
              }
            }
          }
#pragma unroll
          for (int q = 0; q < R; ++q) {
            if (rb + q >= hi) break;
            float mx = ls[q];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float w = (ls[q] == -INFINITY) ? 0.f : ex2(ls[q] - mx);
            float wsum = w;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
            float acc[E];
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
            for (int s = 0; s < kMaxClusterSplits; ++s) {
              if (s < S) {
                const float ws = __shfl_sync(0xffffffffu, w, s);
                if (ws != 0.f) {  // skipped peers may hold stale, non-finite rows
                  acc[0] += ws * v4[q][s].x;
                  acc[1] += ws * v4[q][s].y;
                  if constexpr (E == 4) {
                    acc[2] += ws * v4[q][s].z;
                    acc[3] += ws * v4[q][s].w;
                  }
                }
              }
            }
            const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
            __nv_bfloat16* dst = p.out + out_row[q] * D + lane * E;
            if constexpr (E == 4) {
              uint2 v;
              v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
              v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
              *reinterpret_cast<uint2*>(dst) = v;
            } else {
              *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            }
            if (lane == 0 && p.lse != nullptr) p.lse[out_row[q]] = (mx + log2f(wsum)) * kLn2;
          }
        }
      } else if (lane == 0) {
        report_error(p.err, SV_DEVERR_TIMEOUT);
      }
      if (r_cta == 0) mark(SV_TRACE_MERGE_DONE);
    }
  }
  }  // row group exists

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) mark(SV_TRACE_EXIT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Merge split partials: O = sum_s w_s O_s / sum_s w_s, w_s = 2^(lse_s - max).
template <int D>
__global__ void __launch_bounds__(256) split_combine_kernel(const __nv_bfloat16* __restrict__ part_o,
                                                            const float* __restrict__ part_lse,
                                                            __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                                            int rows, int splits) {
  constexpr int E = D / 32;  // elements per lane
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, part_lse[static_cast<size_t>(s) * rows + row]);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float ls = part_lse[static_cast<size_t>(s) * rows + row];
    if (ls == -INFINITY) continue;
    const float w = ex2(ls - mx);
    wsum += w;
    const __nv_bfloat16* src = part_o + (static_cast<size_t>(s) * rows + row) * D + lane * E;
    if constexpr (E == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(src);
      acc[0] += w * __uint_as_float(v.x << 16);
      acc[1] += w * __uint_as_float(v.x & 0xFFFF0000u);
      acc[2] += w * __uint_as_float(v.y << 16);
      acc[3] += w * __uint_as_float(v.y & 0xFFFF0000u);
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(src);
      acc[0] += w * __uint_as_float(v << 16);
      acc[1] += w * __uint_as_float(v & 0xFFFF0000u);
    }
  }
  const float inv = 1.f / wsum;
  __nv_bfloat16* dst = out + static_cast<size_t>(row) * D + lane * E;
  if constexpr (E == 4) {
    uint2 w;
    w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lse != nullptr && lane == 0) lse[row] = (mx + log2f(wsum)) * kLn2;
}

// ------------------------------------------------------------------ host

std::mutex g_trace_mu;
unsigned long long* g_trace = nullptr;
long long g_trace_ctas = 0;

struct Plan {
  int group;
  int groups_per_seq;
  int splits;
  int mode;
  size_t workspace;
};

sv_status validate(const sv_attn_params* p) {
  if (p == nullptr) return SV_ERR_INVALID_ARG;
  if (p->batch < 1 || p->num_q_heads < 1 || p->num_kv_heads < 1 || p->total_nodes < 0 || p->max_nodes < 1 ||
      p->max_pages_per_seq < 1 || p->num_pages < 1 || p->num_splits < 0 || p->max_kv_pages < 0 ||
      p->split_reduce < 0 || p->split_reduce > 2)
    return SV_ERR_INVALID_ARG;
  if (p->num_q_heads % p->num_kv_heads != 0) return SV_ERR_INVALID_ARG;
  const int G = p->num_q_heads / p->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return SV_ERR_UNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 128) return SV_ERR_UNSUPPORTED;
  if (p->page_size != 16) return SV_ERR_UNSUPPORTED;
  if (p->max_nodes > kMaxNodes) return SV_ERR_UNSUPPORTED;
  if (p->num_splits > kMaxSplits) return SV_ERR_UNSUPPORTED;
  if (p->split_reduce == 1 && p->num_splits > kMaxClusterSplits) return SV_ERR_UNSUPPORTED;
  if (!p->q || !p->tree_k || !p->tree_v || !p->k_cache || !p->v_cache || !p->block_table || !p->ctx_lens ||
      !p->cu_nodes || !p->parents || !p->out)
    return SV_ERR_INVALID_ARG;
  if ((p->kv_pages == nullptr) != (p->cu_kv_pages == nullptr)) return SV_ERR_INVALID_ARG;
  if (!aligned16(p->q) || !aligned16(p->tree_k) || !aligned16(p->tree_v) || !aligned16(p->k_cache) ||
      !aligned16(p->v_cache) || !aligned16(p->out))
    return SV_ERR_INVALID_ARG;
  if (static_cast<long long>(p->batch) * p->num_kv_heads * ((p->max_nodes * G + kCtaRows - 1) / kCtaRows) > 65535)
    return SV_ERR_UNSUPPORTED;
  return SV_OK;
}

template <int D>
void launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attrs, dim3 grid, int cluster, cudaStream_t s) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = grid;
  cfg->blockDim = dim3(kThreads, 1, 1);
  cfg->dynamicSmemBytes = Cfg<D>::kSmemBytes;
  cfg->stream = s;
  int n = 0;
  attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = cluster;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg->attrs = attrs;
  cfg->numAttrs = n;
}

// One-time per-device kernel attributes (dynamic smem, cluster size > 8).
template <int D>
bool configure_kernel() {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && done[dev]) return true;
  if (cudaFuncSetAttribute(tree_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<D>::kSmemBytes) != cudaSuccess)
    return false;
  if (cudaFuncSetAttribute(tree_attention_kernel<D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
      cudaSuccess)
    return false;
  if (dev < 64) done[dev] = true;
  return true;
}

// Co-resident clusters of `size` CTAs at this kernel's footprint (cached per
// device); 0 when they cannot be scheduled or the query fails.
template <int D>
int max_active_clusters(int size) {
  static std::mutex mu;
  static int cache[64][kMaxClusterSplits + 1];
  static bool init = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (auto& row : cache)
      for (int& v : row) v = -1;
    init = true;
  }
  if (cache[dev][size] >= 0) return cache[dev][size];
  int n = 0;
  if (configure_kernel<D>()) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attrs[2];
    launch_config<D>(&cfg, attrs, dim3(size, 1, 1), size, nullptr);
    if (cudaOccupancyMaxActiveClusters(&n, tree_attention_kernel<D>, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cache[dev][size] = n;
  return n;
}

int active_clusters(int head_dim, int size) {
  return head_dim == 128 ? max_active_clusters<128>(size) : max_active_clusters<64>(size);
}

// Split count and merge mode from a small cost model in units of one KV tile
// of work: a CTA costs its share of tiles plus a fixed prologue/epilogue;
// waves come from how many CTAs (or clusters) are co-resident; an on-chip
// merge costs a little per CTA, a global merge costs partial writes plus a
// second kernel.
void choose_splits(const sv_attn_params* p, int sms, int groups_per_seq, int* splits, int* mode) {
  const long long units = static_cast<long long>(p->batch) * p->num_kv_heads * groups_per_seq;
  const int pages = p->kv_pages ? p->max_kv_pages : p->max_pages_per_seq;
  const int tiles = (pages + kPagesPerTile - 1) / kPagesPerTile + 1;
  // merge costs measured on GB300 (in tiles of work): the in-cluster merge is
  // latency-bound (~5 us); partial writes ~1 tile; the combine kernel ~2
  const double c_cta = 1.5, c_red = 4.0, c_part = 1.0, c_comb = 2.0;
  auto cost_cluster = [&](int s) -> double {
    const int act = active_clusters(p->head_dim, s);
    if (act <= 0) return 1e300;
    const long long waves = (units + act - 1) / act;
    return static_cast<double>(waves) * (static_cast<double>((tiles + s - 1) / s) + c_cta + c_red);
  };
  auto cost_global = [&](int s) -> double {
    const long long waves = (units * s + sms - 1) / sms;
    return static_cast<double>(waves) * (static_cast<double>((tiles + s - 1) / s) + c_cta + c_part) + c_comb +
           0.05 * s;
  };
  if (p->num_splits > 0) {
    *splits = p->num_splits;
    if (*splits == 1) *mode = kReduceNone;
    else if (p->split_reduce == 2) *mode = kReduceGlobal;
    else if (p->split_reduce == 1) *mode = kReduceCluster;
    else *mode = (*splits <= 8 || (*splits <= kMaxClusterSplits && sms > 0 && active_clusters(p->head_dim, *splits) > 0))
                     ? kReduceCluster : kReduceGlobal;
    return;
  }
  const long long waves1 = (units + sms - 1) / sms;
  double best = static_cast<double>(waves1) * (tiles + c_cta);
  *splits = 1;
  *mode = kReduceNone;
  for (int s = 2; s <= kMaxSplits && s <= tiles; ++s) {
    if (p->split_reduce != 2 && s <= kMaxClusterSplits) {
      const double c = cost_cluster(s);
      if (c < best - 1e-9) {
        best = c;
        *splits = s;
        *mode = kReduceCluster;
      }
    }
    if (p->split_reduce != 1) {
      const double c = cost_global(s);
      if (c < best - 1e-9) {
        best = c;
        *splits = s;
        *mode = kReduceGlobal;
      }
    }
  }
}

sv_status make_plan(const sv_attn_params* p, Plan* plan) {
  sv_status st = validate(p);
  if (st != SV_OK) return st;
  plan->group = p->num_q_heads / p->num_kv_heads;
  plan->groups_per_seq = (p->max_nodes * plan->group + kCtaRows - 1) / kCtaRows;
  int sms = 0;
  if (p->num_splits == 0 || (p->num_splits > 8 && p->split_reduce == 0)) {
    sms = device_sm_count();
    if (sms <= 0) return SV_ERR_CUDA;
  }
  choose_splits(p, sms, plan->groups_per_seq, &plan->splits, &plan->mode);
  size_t ws = kWorkspaceHeader;
  if (plan->mode != kReduceNone) {
    const size_t rows = static_cast<size_t>(p->total_nodes) * p->num_q_heads;
    ws += align_up(static_cast<size_t>(plan->splits) * rows * p->head_dim * 2, 256);  // bf16 O / l
    ws += align_up(static_cast<size_t>(plan->splits) * rows * sizeof(float), 256);   // log2-sum-exp
  }
  plan->workspace = ws;
  return SV_OK;
}

template <int D>
sv_status launch(const sv_attn_params* p, const Plan& plan, cudaStream_t stream) {
  if (!configure_kernel<D>()) return SV_ERR_CUDA;
  const int G = plan.group;
  const cuuint64_t T = static_cast<cuuint64_t>(p->total_nodes);
  const cuuint64_t Hq = p->num_q_heads, Hkv = p->num_kv_heads, Dd = D, P = p->page_size;
  CUtensorMap tm_q, tm_kc, tm_vc, tm_tk, tm_tv;
  {
    const cuuint64_t dims[3] = {Dd, Hq, T};
    const cuuint64_t strides[2] = {Dd * 2, Hq * Dd * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(kTileRows / G)};
    if (encode_tiled(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p->q), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B) != CUDA_SUCCESS)
      return SV_ERR_CUDA;
  }
  {
    const cuuint64_t dims[4] = {Dd, P, Hkv, static_cast<cuuint64_t>(p->num_pages)};
    const cuuint64_t strides[3] = {Dd * 2, P * Dd * 2, Hkv * P * Dd * 2};
    const cuuint32_t box[4] = {64, 16, 1, 1};
    if (encode_tiled(&tm_kc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(p->k_cache), dims, strides,
                     box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS)
      return SV_ERR_CUDA;
    if (encode_tiled(&tm_vc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(p->v_cache), dims, strides,
                     box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS)
      return SV_ERR_CUDA;
  }
  {
    const cuuint64_t dims[3] = {Dd, Hkv, T};
    const cuuint64_t strides[2] = {Dd * 2, Hkv * Dd * 2};
    const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kBlockN)};
    if (encode_tiled(&tm_tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p->tree_k), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B) != CUDA_SUCCESS)
      return SV_ERR_CUDA;
    if (encode_tiled(&tm_tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p->tree_v), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B) != CUDA_SUCCESS)
      return SV_ERR_CUDA;
  }
  uint8_t* ws = static_cast<uint8_t*>(p->workspace);
  Params kp;
  kp.block_table = p->block_table;
  kp.ctx_lens = p->ctx_lens;
  kp.cu_nodes = p->cu_nodes;
  kp.parents = p->parents;
  kp.kv_pages = p->kv_pages;
  kp.cu_kv_pages = p->cu_kv_pages;
  kp.out = static_cast<__nv_bfloat16*>(p->out);
  kp.lse = p->lse;
  kp.err = reinterpret_cast<int*>(ws);
  {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    kp.trace = g_trace;
    kp.trace_ctas = g_trace_ctas;
  }
  const size_t rows = static_cast<size_t>(p->total_nodes) * p->num_q_heads;
  kp.part_o = nullptr;
  kp.part_lse = nullptr;
  if (plan.mode != kReduceNone) {
    kp.part_o = reinterpret_cast<__nv_bfloat16*>(ws + kWorkspaceHeader);
    kp.part_lse = reinterpret_cast<float*>(ws + kWorkspaceHeader +
                                           align_up(static_cast<size_t>(plan.splits) * rows * D * 2, 256));
  }
  kp.num_q_heads = p->num_q_heads;
  kp.group = G;
  kp.num_pages = p->num_pages;
  kp.max_pages_per_seq = p->max_pages_per_seq;
  kp.num_splits = plan.splits;
  kp.reduce_mode = plan.mode;
  kp.total_nodes = p->total_nodes;
  kp.groups_per_seq = plan.groups_per_seq;
  const float scale = (p->sm_scale > 0.f) ? p->sm_scale : 1.0f / sqrtf(static_cast<float>(D));
  kp.scale_log2 = scale * 1.4426950408889634f;

  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attrs[2];
  launch_config<D>(&cfg, attrs, dim3(plan.splits, p->num_kv_heads * plan.groups_per_seq, p->batch),
                   plan.mode == kReduceCluster ? plan.splits : 1, stream);
  if (cudaLaunchKernelEx(&cfg, tree_attention_kernel<D>, tm_q, tm_kc, tm_vc, tm_tk, tm_tv, kp) != cudaSuccess)
    return SV_ERR_CUDA;
  if (plan.mode == kReduceGlobal) {
    const int blocks = static_cast<int>((rows * 32 + 255) / 256);
    split_combine_kernel<D><<<blocks, 256, 0, stream>>>(kp.part_o, kp.part_lse, kp.out, p->lse,
                                                         static_cast<int>(rows), plan.splits);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  }
  return SV_OK;
}

}  // namespace attn
}  // namespace sv

extern "C" {

sv_status sv_tree_attention_workspace_size(const sv_attn_params* params, size_t* bytes) {
  if (bytes == nullptr) return SV_ERR_INVALID_ARG;
  sv::attn::Plan plan;
  const sv_status st = sv::attn::make_plan(params, &plan);
  if (st != SV_OK) return st;
  *bytes = plan.workspace;
  return SV_OK;
}

sv_status sv_set_trace_buffer(void* buffer, size_t bytes) {
  std::lock_guard<std::mutex> lock(sv::attn::g_trace_mu);
  if (buffer == nullptr) {
    sv::attn::g_trace = nullptr;
    sv::attn::g_trace_ctas = 0;
    return SV_OK;
  }
  if ((reinterpret_cast<uintptr_t>(buffer) & 7u) != 0) return SV_ERR_INVALID_ARG;
  sv::attn::g_trace = static_cast<unsigned long long*>(buffer);
  sv::attn::g_trace_ctas = static_cast<long long>(bytes / (kSvTraceSlots * sizeof(unsigned long long)));
  return SV_OK;
}

sv_status sv_tree_attention_plan(const sv_attn_params* params, int* num_splits, int* split_reduce) {
  if (num_splits == nullptr || split_reduce == nullptr) return SV_ERR_INVALID_ARG;
  sv::attn::Plan plan;
  const sv_status st = sv::attn::make_plan(params, &plan);
  if (st != SV_OK) return st;
  *num_splits = plan.splits;
  *split_reduce = plan.mode;
  return SV_OK;
}

sv_status sv_tree_attention(const sv_attn_params* params, sv_stream_t stream) {
  sv::attn::Plan plan;
  const sv_status st = sv::attn::make_plan(params, &plan);
  if (st != SV_OK) return st;
  if (params->workspace == nullptr || params->workspace_bytes < plan.workspace) return SV_ERR_WORKSPACE;
  if (params->total_nodes == 0) return SV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (params->head_dim == 128) return sv::attn::launch<128>(params, plan, s);
  return sv::attn::launch<64>(params, plan, s);
}

}  // extern "C"
