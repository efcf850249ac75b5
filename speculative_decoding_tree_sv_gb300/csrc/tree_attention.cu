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
// Design (one CTA per (KV split, KV head x 128-row tile, sequence)):
//   * The M dimension of the contraction is (tree node x query head of the
//     GQA group): rows r = node * G + g, one 128-row tile per CTA.
//   * Context K/V pages (16 tokens, head-major inside a page) are gathered
//     with TMA, eight pages (128 keys) per tile, 128-byte swizzled, into
//     rings of K and V stages.  The tree's own K/V form one extra tile.
//   * The two row tiles of a (sequence, KV head) form a two-CTA cluster and
//     read every K/V tile once: each CTA requests half of its pages with
//     cluster multicast, so the tile lands in both CTAs' shared memory, and
//     a stage is refilled only after both CTAs have released it.
//   * Q lives in TMEM (the softmax warps load their rows and store them
//     there), so shared memory holds only K and V stages: the loaded-DRAM
//     latency times the bandwidth a CTA needs is what the rings must cover.
//   * tcgen05.mma computes S = Q K^T (Q from TMEM, K K-major in smem) into
//     one of two TMEM score buffers, so the tensor core computes the next
//     tile's scores while the softmax warps work on the current ones.
//     Softmax reads S with tcgen05.ld (one row per thread), applies the mask
//     and an online, lazily rescaled base-2 softmax (packed two-lane fp32
//     arithmetic), and writes P as bf16 back into the score columns;
//     tcgen05.mma accumulates O += P V (P from TMEM, V MN-major in smem).
//     TMEM columns: S0, S1, O, Q.  MMA order: S0 S1 | PV0 S2 | PV1 S3 | ...
//   * Warp roles: warp 0 loads the K tiles, warp 3 the V tiles, warp 2
//     resolves page ids ahead of them, warp 1 runs the MMA schedule
//     (converged; one elected lane issues each MMA and commit), warps 4-7
//     load Q, run the softmax and the epilogue.
//   * KV splits write partials (O / l in bf16 and log2-sum-exp) to the
//     workspace; a combine kernel merges them.
//   * Launches allow programmatic dependent launch: the prologue (barriers,
//     TMEM, descriptor prefetch) runs before the wait on the previous grid.
#include <math.h>

#include <mutex>

#include "sv_device.cuh"

namespace sv {
namespace attn {

constexpr int kThreads = 256;   // 4 control warps + one softmax warpgroup
constexpr int kBlockN = 128;    // keys per tile (8 pages)
constexpr int kTileRows = 128;  // rows per CTA (one M tile)
constexpr int kPagesPerTile = kBlockN / 16;
// Page ids of the next tiles travel from the warp that resolves them to the
// two loader warps through a small ring in shared memory.
constexpr int kIdSlots = 8;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: defer O rescale until max grows by 2^8
constexpr float kLn2 = 0.69314718055994530942f;
constexpr uint16_t kPairMask = 0x3;  // both CTAs of a two-CTA cluster

enum ReduceMode : int { kReduceNone = 0, kReduceGlobal = 2 };

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;                  // 128-byte column halves
  // K stages return to the loader as soon as their QK^T is done, V stages
  // only after PV: the V ring is the deeper one
  static constexpr int kKStages = (D == 128) ? 3 : 5;
  static constexpr int kVStages = (D == 128) ? 4 : 6;
  static constexpr uint32_t kHalfBytes = 128u * 128u;     // 128 rows x 128 B
  static constexpr uint32_t kTileBytes = kTileRows * D * 2;  // K and V tiles alike
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kVStages * kTileBytes;
  static constexpr uint32_t kBarBytes = 1024;
  static constexpr uint32_t kOffIds = kOffBar + 512;      // int32 [kIdSlots][kPagesPerTile]
  static constexpr uint32_t kOffParents = kOffBar + kBarBytes;  // int32 [kMaxNodes]
  static constexpr uint32_t kSmemBytes = kOffParents + kMaxNodes * 4 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
  static constexpr uint32_t kColQ = kColO + D;  // Q as bf16 pairs: D / 2 columns
  // epilogue staging of bf16 output rows (one padded row per softmax thread)
  // over the K stages once every MMA and load is done
  static constexpr uint32_t kStageStride = D * 2 + 16;
  static constexpr uint32_t kOffStage = 0;
  static_assert(kOffStage + kTileRows * kStageStride <= kOffBar, "staging must fit below the barriers");
  static_assert((1 + 2 * kKStages + 2 * kVStages + 7 + 2 * kIdSlots) * 8 + 12 <= 512,
                "barriers must fit below the id ring");
  static_assert(512 + kIdSlots * kPagesPerTile * 4 <= kBarBytes - 8, "id ring must fit below the trace word");
  static_assert(kColQ + D / 2 <= kTmemCols, "TMEM columns");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct Params {
  const int* block_table;
  const int* ctx_lens;
  const int* cu_nodes;
  const int* parents;
  const int* kv_pages;
  const int* cu_kv_pages;
  const __nv_bfloat16* q;
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
  int max_nodes;
  int num_splits;
  int reduce_mode;
  int early_ctx;  // read index arrays and context pages before the wait on the preceding grid
  int early_trigger;  // let the dependent grid launch at once (small grids: the SMs are free)
  int total_nodes;
  int row_tiles;  // 128-row tiles per (sequence, KV head); even when paired
  int paired;     // row tiles 2q, 2q+1 form a two-CTA cluster sharing K/V
  float scale_log2;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    tree_attention_kernel(const __grid_constant__ CUtensorMap tm_kc,
                          const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_tk,
                          const __grid_constant__ CUtensorMap tm_tv, const __grid_constant__ Params p) {
  using C = Cfg<D>;
  constexpr int NSK = C::kKStages;
  constexpr int NSV = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int split = blockIdx.x;
  const int kh = blockIdx.y / p.row_tiles;
  const int rt = blockIdx.y % p.row_tiles;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const bool paired = p.paired != 0;
  const uint32_t rank = paired ? cluster_ctarank() : 0u;  // equals rt & 1 when paired
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
  uint64_t* q_full = bars;          // Q rows stored in TMEM by the softmax warps
  uint64_t* k_full = bars + 1;      // [NSK]
  uint64_t* v_full = k_full + NSK;  // [NSV]
  uint64_t* k_empty = v_full + NSV; // [NSK] released by this CTA's MMAs (and the peer's when paired)
  uint64_t* v_empty = k_empty + NSK;  // [NSV]
  uint64_t* s_full = v_empty + NSV;   // [2] scores of a buffer ready
  uint64_t* p_full = s_full + 2;      // [2] probabilities of a buffer written
  uint64_t* pv_done = p_full + 2;     // one phase per tile: O += P V finished
  uint64_t* o_final = pv_done + 1;
  uint64_t* drain = o_final + 1;
  uint64_t* ids_full = drain + 1;             // [kIdSlots] page ids of a tile written
  uint64_t* ids_empty = ids_full + kIdSlots;  // [kIdSlots] both loaders read them
  int* ids = reinterpret_cast<int*>(smem + C::kOffIds);
  int* par_s = reinterpret_cast<int*>(smem + C::kOffParents);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ids_empty + kIdSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never_set = abort_flag + 1;  // drains wait on copies even after an abort

  // ---- prologue that reads no input: it may overlap the previous grid
  if (threadIdx.x == 0) {
    mbar_init(q_full, kTileRows);
    for (int i = 0; i < NSK; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, paired ? 2 : 1);
    }
    for (int i = 0; i < NSV; ++i) {
      mbar_init(v_full + i, 1);
      mbar_init(v_empty + i, paired ? 2 : 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full + t, 1);
      mbar_init(p_full + t, kTileRows);
    }
    mbar_init(pv_done, 1);
    mbar_init(o_final, 1);
    mbar_init(drain, 1);
    for (int i = 0; i < kIdSlots; ++i) {
      mbar_init(ids_full + i, 1);
      mbar_init(ids_empty + i, 2);
    }
    *abort_flag = 0;
    *never_set = 0;
    fence_mbar_init();
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
  // both CTAs of a pair reach this point: the peer's barriers are initialised
  // before any multicast copy or remote arrive can reach them
  if (paired) cluster_sync_all();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) mark(SV_TRACE_PROLOGUE);
  // Everything below that reads what the preceding grid may write (Q, the
  // tree's K/V) or writes what it may read (outputs, workspace) waits for it
  // first; with early_ctx the index arrays and context pages are read
  // before that wait.
  if (!p.early_ctx) griddep_wait();
  // Without a split merge the next grid is the next attention call: let it
  // start its prologue now.  With one, the next grid is the combine kernel,
  // which is only useful once the partials are written (signalled at exit),
  // unless the grid is small enough to leave most SMs to it (its own wait
  // on this grid keeps it correct either way).
  if (p.reduce_mode == kReduceNone || p.early_trigger) griddep_launch_dependents();
  if (threadIdx.x == 0) mark(SV_TRACE_INPUTS);
  // the z-th longest sequence (batches of up to 64; the index itself beyond)
  const int b = longest_first_seq(blockIdx.z, gridDim.z, p.ctx_lens, p.cu_kv_pages);
  // With the full context, tiles are dealt to the splits in turn (split s
  // takes tiles s, s + S, ...), so a split's first tile is tile s whatever
  // the context's length and the page-id warp requests its block-table
  // entries before the length arrives.  A partial list keeps contiguous
  // ranges (its ids come from the list itself, one read later anyway).
  int spec_phys = 0;
  bool spec_ok = false;
  if (warp == 2 && lane < kPagesPerTile && p.kv_pages == nullptr) {
    const int e = split * kPagesPerTile + lane;
    if (e < p.max_pages_per_seq) {
      spec_phys = p.block_table[static_cast<size_t>(b) * p.max_pages_per_seq + e];
      spec_ok = true;
    }
  }

  const int n0 = p.cu_nodes[b];
  const int N = p.cu_nodes[b + 1] - n0;
  const int L = p.ctx_lens[b];
  if (threadIdx.x == 0 && split == 0 && rt == 0 && kh == 0 && (N < 1 || N > p.max_nodes))
    report_error(p.err, SV_DEVERR_BAD_TREE);
  const int rows_total = N * G;
  const int row0 = rt * kTileRows;
  // a pair works when either of its tiles has rows (uniform over the pair)
  const int pair_row0 = paired ? (rt & ~1) * kTileRows : row0;
  if (pair_row0 < rows_total) {
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
  const bool dealt = !partial;  // tiles dealt in turn (full context) or contiguous (partial list)
  const int jb = dealt ? split : static_cast<int>(static_cast<long long>(split) * t_all / p.num_splits);
  const int jstep = dealt ? p.num_splits : 1;
  const int ntiles = dealt ? (split < t_all ? (t_all - 1 - split) / p.num_splits + 1 : 0)
                           : static_cast<int>(static_cast<long long>(split + 1) * t_all / p.num_splits) - jb;
  const bool owns_tree = ntiles > 0 && jb + (ntiles - 1) * jstep == t_all - 1;  // the last tile is the tree's
  const bool work = ntiles > 0;  // uniform over the pair

  if (!work && p.reduce_mode == kReduceGlobal) {
    // empty split: publish an empty partial for our rows
    griddep_wait();
    if (threadIdx.x < kTileRows) {
      const int row = row0 + threadIdx.x;
      if (row < rows_total) {
        const int node = row / G, g = row - (row / G) * G;
        p.part_lse[(static_cast<size_t>(split) * p.total_nodes + n0 + node) * p.num_q_heads + kh * G + g] =
            -INFINITY;
      }
    }
  } else if (warp < 4) {
    if (work && warp == 2) {
      // ------------------------------------------------------------ page ids
      // Resolves each context tile's eight page ids (partial list, then block
      // table, both range-checked) into the id ring, up to kIdSlots tiles
      // ahead of the loaders.
      bool ok = true;
      for (int it = 0; it < ntiles; ++it) {
        const int j = jb + it * jstep;
        const int sl = it % kIdSlots;
        if (it >= kIdSlots) {
          int w = (lane == 0) ? (mbar_wait(ids_empty + sl, ((it / kIdSlots) & 1) ^ 1u, abort_flag) ? 1 : 0) : 0;
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
        }
        if (j < t_ctx && lane < kPagesPerTile) {
          const int ps = min(j * kPagesPerTile + lane, n_pages - 1);  // ragged tail repeats the last page
          int lp = partial ? p.kv_pages[kvp0 + ps] : ps;
          if (lp < 0 || lp >= p.max_pages_per_seq) {
            report_error(p.err, SV_DEVERR_BAD_PAGE);
            lp = 0;
          }
          int phys = (it == 0 && spec_ok && lp == split * kPagesPerTile + lane)
                         ? spec_phys
                         : p.block_table[static_cast<size_t>(b) * p.max_pages_per_seq + lp];
          if (phys < 0 || phys >= p.num_pages) {
            report_error(p.err, SV_DEVERR_BAD_PAGE);
            phys = 0;
          }
          ids[sl * kPagesPerTile + lane] = phys;
        }
        __syncwarp();
        if (lane == 0) {
          if (it == 0) mark(SV_TRACE_FIRST_IDS);
          mbar_arrive(ids_full + sl);
        }
      }
      if (!ok && lane == 0) {
        report_error(p.err, SV_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
    } else if (work && (warp == 0 || warp == 3)) {
      // ------------------------------------------------------------ loaders
      // warp 0 loads the K tiles, warp 3 the V tiles, each as far ahead as
      // its ring allows.  When paired, each CTA requests four of a
      // tile's eight pages (and one column half of the tree tile) with
      // multicast to both CTAs; every CTA's full barrier expects the whole
      // tile.
      const bool is_k = warp == 0;
      const CUtensorMap* tm_cache = is_k ? &tm_kc : &tm_vc;
      const CUtensorMap* tm_tree = is_k ? &tm_tk : &tm_tv;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* ring = smem + (is_k ? C::kOffK : C::kOffV);
      const int NS = is_k ? NSK : NSV;
      const int lane_lo = paired ? 4 * static_cast<int>(rank) : 0;
      const int lane_hi = paired ? lane_lo + 4 : kPagesPerTile;
      int issued = 0;
      // one tile into the ring; false when a bounded wait ran out
      auto load_tile = [&](int it) -> bool {
        const int j = jb + it * jstep;
        const int st = it % NS;
        const uint32_t ph = (it / NS) & 1;
        const int sl = it % kIdSlots;
        const bool ctx = j < t_ctx;
        {
          int w = (lane == 0) ? (mbar_wait(ids_full + sl, (it / kIdSlots) & 1, abort_flag) ? 1 : 0) : 0;
          if (!__shfl_sync(0xffffffffu, w, 0)) return false;
        }
        const int phys = (ctx && lane < kPagesPerTile) ? ids[sl * kPagesPerTile + lane] : 0;
        if (it >= NS) {
          int w = (lane == 0) ? (mbar_wait(empty + st, ph ^ 1u, abort_flag) ? 1 : 0) : 0;
          if (!__shfl_sync(0xffffffffu, w, 0)) return false;
        }
        if (lane == 0) mbar_arrive_expect_tx(full + st, C::kTileBytes);
        __syncwarp();
        uint8_t* dst = ring + st * C::kTileBytes;
        if (ctx) {
          if (lane >= lane_lo && lane < lane_hi) {
            for (int h = 0; h < C::kHalves; ++h) {
              if (paired)
                tma_load_4d_mc(dst + h * C::kHalfBytes + lane * 2048, tm_cache, full + st, h * 64, 0, kh, phys,
                               kPairMask);
              else
                tma_load_4d(dst + h * C::kHalfBytes + lane * 2048, tm_cache, full + st, h * 64, 0, kh, phys);
            }
          }
        } else if (lane == 0) {
          for (int h = 0; h < C::kHalves; ++h) {
            if (!paired)
              tma_load_3d(dst + h * C::kHalfBytes, tm_tree, full + st, h * 64, kh, n0);
            else if (C::kHalves == 2 ? h == static_cast<int>(rank) : rank == 0u)
              tma_load_3d_mc(dst + h * C::kHalfBytes, tm_tree, full + st, h * 64, kh, n0, kPairMask);
          }
        }
        issued = it + 1;
        __syncwarp();
        if (lane == 0) mbar_arrive(ids_empty + sl);
        return true;
      };
      bool ok = true;
      int it = 0;
      if (p.early_ctx) {
        // Context pages are not written by the preceding grid: the first
        // ring's worth of them is requested before waiting for it.
        for (; ok && it < ntiles && it < NS && jb + it * jstep < t_ctx; ++it) ok = load_tile(it);
      }
      griddep_wait();  // the tree's K/V come from the preceding grid
      for (; ok && it < ntiles; ++it) ok = load_tile(it);
      if (!ok && lane == 0) {
        // Timed out: stop the other roles, then let our copies land before exit.
        report_error(p.err, SV_DEVERR_TIMEOUT);
        *abort_flag = 1;
        for (int i = max(0, issued - NS); i < issued; ++i) mbar_wait(full + (i % NS), (i / NS) & 1, never_set);
      }
    } else if (work && warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs the schedule, so descriptors and loop state stay
      // warp-uniform; one elected lane issues each MMA and commit.  (Issuing
      // from a lane-0-only branch cost about three times the MMA's own time
      // per instruction.)
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kBlockN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
      const uint32_t k_base = smem_u32(smem + C::kOffK);
      const uint32_t v_base = smem_u32(smem + C::kOffV);
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
      };
      auto commit = [&](uint64_t* bar) {
        if (elect_one()) umma_commit(bar);
        __syncwarp();
      };
      // S = Q K^T: Q (bf16 pairs) from TMEM, K K-major from shared memory
      auto issue_qk = [&](int buf, int kst) {
        const uint32_t d = tmem + (buf ? C::kColS1 : C::kColS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
          const uint64_t bdesc = smem_desc_sw128(k_base + kst * C::kTileBytes + off, 16, 1024);
          if (elect_one()) umma_ts(d, tmem + C::kColQ + kk * 8, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
          __syncwarp();
        }
      };
      // O += P V: P (bf16 pairs) in the score buffer's first columns
      auto issue_pv = [&](int buf, int vst, bool accumulate) {
        const uint32_t d = tmem + C::kColO;
        const uint32_t a = tmem + (buf ? C::kColS1 : C::kColS0);
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(v_base + vst * C::kTileBytes + kk * 2048, C::kHalfBytes, 1024);
          if (elect_one()) umma_ts(d, a + kk * 8, bdesc, idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
          __syncwarp();
        }
      };
      // A stage goes back to the loaders of both CTAs of a pair once this
      // CTA's MMAs have read it.  The last stages of a ring are never
      // refilled, so they are not released: no arrive is left in flight
      // towards the peer when the CTAs finish.
      auto release = [&](uint64_t* bar, int it, int ns) {
        if (it + ns < ntiles) {
          if (elect_one()) {
            if (paired) umma_commit_mc(bar, kPairMask);
            else umma_commit(bar);
          }
          __syncwarp();
        }
      };
      bool ok = wait_all(q_full, 0);
      // scores of the first two tiles, one per buffer
      for (int it = 0; ok && it < 2 && it < ntiles; ++it) {
        if (!wait_all(k_full + it % NSK, (it / NSK) & 1)) { ok = false; break; }
        tc_fence_after();
        if (it == 0 && lane == 0) mark(SV_TRACE_FIRST_MMA);
        issue_qk(it, it % NSK);
        commit(s_full + it);
        release(k_empty + it % NSK, it, NSK);
      }
      for (int it = 0; ok && it < ntiles; ++it) {
        const int buf = it & 1;
        const int vst = it % NSV;
        if (!wait_all(v_full + vst, (it / NSV) & 1)) { ok = false; break; }
        if (!wait_all(p_full + buf, (it >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        issue_pv(buf, vst, it > 0);
        commit(pv_done);
        release(v_empty + vst, it, NSV);
        // the next scores of this buffer overwrite P(it) after PV(it) has
        // read it: tcgen05 MMAs of one thread execute in issue order
        const int nx = it + 2;
        if (nx < ntiles) {
          const int kst = nx % NSK;
          if (!wait_all(k_full + kst, (nx / NSK) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_qk(buf, kst);
          commit(s_full + buf);
          release(k_empty + kst, nx, NSK);
        }
      }
      if (ok) {
        commit(o_final);
      } else {
        if (lane == 0) {
          report_error(p.err, SV_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        commit(drain);  // let issued MMAs finish before TMEM is freed
        __all_sync(0xffffffffu, mbar_wait(drain, 0, never_set));
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int qw = warp - 4;
    const int r = qw * 32 + lane;  // TMEM lane = row of the tile
    const int row = row0 + r;
    const bool row_exists = row < rows_total;
    // A warp whose 32 rows are all past the tree's rows only keeps the
    // barrier protocol (its S and P columns are never read back into an
    // output), which frees its scheduler's issue slots for the other warps.
    const bool warp_rows = __any_sync(0xffffffffu, row_exists);
    const int node = row / G;
    const int g = row - node * G;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    const size_t orow = static_cast<size_t>(n0 + node) * p.num_q_heads + kh * G + g;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    if (work) {
      // Q: each thread moves its row (zeros past the tree) into TMEM as bf16
      // pairs, the A operand of QK^T
      griddep_wait();  // Q comes from the preceding grid
      {
        const uint4* src = reinterpret_cast<const uint4*>(p.q + orow * D);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t qv[32];
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint4 t = row_exists ? __ldg(src + c * 8 + v) : make_uint4(0u, 0u, 0u, 0u);
            qv[4 * v + 0] = t.x;
            qv[4 * v + 1] = t.y;
            qv[4 * v + 2] = t.z;
            qv[4 * v + 3] = t.w;
          }
          tmem_st32(lane_base + C::kColQ + c * 32, qv);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(q_full);
      }
      // ancestor-or-self bitmask of this row's node (only the split that
      // owns the tree tile needs it): the tree's parents are staged in shared
      // memory with one coalesced load, then each row walks its chain there
      uint32_t anc0 = 0, anc1 = 0, anc2 = 0, anc3 = 0;
      if (owns_tree) {
        for (int i = r; i < N && i < kMaxNodes; i += kTileRows) par_s[i] = p.parents[n0 + i];
        named_barrier(1, kTileRows);
        if (row_exists) {
          int c = node;
          for (int step = 0; step < kMaxNodes && c >= 0 && c < kMaxNodes && c < N; ++step) {
            const uint32_t bit = 1u << (c & 31);
            if ((c >> 5) == 0) anc0 |= bit;
            else if ((c >> 5) == 1) anc1 |= bit;
            else if ((c >> 5) == 2) anc2 |= bit;
            else anc3 |= bit;
            if (c == 0) break;
            const int pc = par_s[c];
            if (pc < 0 || pc >= c) {
              report_error(p.err, SV_DEVERR_BAD_PARENT);
              break;
            }
            c = pc;
          }
        }
        if (r == 0) mark(SV_TRACE_TREE_MASK);
      }
      for (int it = 0; it < ntiles; ++it) {
        const int j = jb + it * jstep;
        const int buf = it & 1;
        const uint32_t col_s = buf ? C::kColS1 : C::kColS0;
        // warp-uniform outcome: the TMEM loads below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(s_full + buf, (it >> 1) & 1, abort_flag))) { ok = false; break; }
        if (!warp_rows) {
          mbar_arrive(p_full + buf);
          continue;
        }
        tc_fence_after();
        if (it == 0 && r == 0) mark(SV_TRACE_FIRST_S);
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
        // instructions: the whole warp takes it when any row needs it (rows
        // that do not are scaled by 1).  O holds tiles up to it - 1; the PV
        // of tile it - 1 may still be running, so wait for it first.
        if (it > 0 && __any_sync(0xffffffffu, grow)) {
          if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (it - 1) & 1, abort_flag))) { ok = false; break; }
          tc_fence_after();
          const float f = grow ? ex2(m_run - m_new) : 1.f;
          l_run *= f;
          const uint64_t f2 = f2_pack(f, f);
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            tmem_ld32(lane_base + C::kColO + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              const uint64_t v = f2_mul(f2_pack(__uint_as_float(o[k]), __uint_as_float(o[k + 1])), f2);
              o[k] = static_cast<uint32_t>(v);
              o[k + 1] = static_cast<uint32_t>(v >> 32);
            }
            tmem_st32(lane_base + C::kColO + c * 32, o);
          }
          tmem_st_wait();
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
          const uint64_t bb = f2_fma(f2_pack(__uint_as_float(sr[k + 2]), __uint_as_float(sr[k + 3])), sc2, nm2);
          const float p0 = ex2(f2_lo(a)), p1 = ex2(f2_hi(a));
          const float p2 = ex2(f2_lo(bb)), p3 = ex2(f2_hi(bb));
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
        mbar_arrive(p_full + buf);
      }
      if (r == 0) mark(SV_TRACE_LOOP_END);
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_final, 0, abort_flag));
      if (r == 0) mark(SV_TRACE_O_READY);
      if (!ok && lane == 0) {
        report_error(p.err, SV_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
    }

    // ---------------------------------------------------------- epilogue
    griddep_wait();  // outputs and workspace may still be in use by the preceding grid
    const bool have_o = work && ok && warp_rows;  // warp-uniform
    if (have_o) tc_fence_after();
    const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
    const float lse2 = (have_o && l_run > 0.f) ? m_run + log2f(l_run) : -INFINITY;
    // Output rows leave through shared memory: each thread parks its row
    // (one TMEM lane) in a padded staging row over the dead K stages (every
    // MMA and every load has finished once o_final fired), then the warp
    // writes whole rows, lane l moving chunk l, so global stores are
    // coalesced.
    const bool partial_out = p.reduce_mode != kReduceNone;
    if (have_o) {
      uint8_t* stage = smem + C::kOffStage + qw * 32 * C::kStageStride;
      uint8_t* mine = stage + lane * C::kStageStride;
#pragma unroll
      for (int c = 0; c < D / 32; c += 2) {
        uint32_t o[2][32];
        tmem_ld32(lane_base + C::kColO + c * 32, o[0]);
        tmem_ld32(lane_base + C::kColO + (c + 1) * 32, o[1]);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o[h][8 * v + 0]) * inv_l, __uint_as_float(o[h][8 * v + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(o[h][8 * v + 2]) * inv_l, __uint_as_float(o[h][8 * v + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(o[h][8 * v + 4]) * inv_l, __uint_as_float(o[h][8 * v + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(o[h][8 * v + 6]) * inv_l, __uint_as_float(o[h][8 * v + 7]) * inv_l);
          reinterpret_cast<uint4*>(mine + (c + h) * 64)[v] = w;
        }
      }
      __syncwarp();
      // rows of D bf16 = D / 8 16-byte chunks; the warp stores 256 / D rows per
      // instruction
      constexpr int kChunks = D / 8;
      constexpr int kRowsPerPass = 32 / kChunks;
      const int wrow0 = row0 + qw * 32;
      const int nrows = min(32, rows_total - wrow0);
      const size_t split_base = partial_out ? static_cast<size_t>(split) * p.total_nodes * p.num_q_heads : 0;
      const long long my_out_row = static_cast<long long>(split_base + orow);  // this lane's row
      __nv_bfloat16* const base = partial_out ? p.part_o : p.out;
      // every shuffle and staging load is issued before the first store
      constexpr int kPasses = 32 / kRowsPerPass;
      uint4 val[kPasses];
      long long gout[kPasses];
#pragma unroll
      for (int i = 0; i < kPasses; ++i) {
        const int rr = i * kRowsPerPass + lane / kChunks;
        gout[i] = __shfl_sync(0xffffffffu, my_out_row, rr);
        val[i] = reinterpret_cast<const uint4*>(stage + rr * C::kStageStride)[lane % kChunks];
      }
#pragma unroll
      for (int i = 0; i < kPasses; ++i) {
        const int rr = i * kRowsPerPass + lane / kChunks;
        if (rr < nrows) reinterpret_cast<uint4*>(base + gout[i] * D)[lane % kChunks] = val[i];
      }
    }
    if (p.reduce_mode == kReduceNone) {
      if (have_o && row_exists && p.lse != nullptr) p.lse[orow] = lse2 * kLn2;
    } else if (row_exists) {
      p.part_lse[static_cast<size_t>(split) * p.total_nodes * p.num_q_heads + orow] = lse2;
    }
    if (r == 0) mark(SV_TRACE_EPILOGUE);
  }
  }  // the pair has rows

  tc_fence_before();
  __syncthreads();
  if (p.reduce_mode != kReduceNone && !p.early_trigger) griddep_launch_dependents();
  // neither CTA of a pair leaves while the other may still address its
  // shared memory (multicast copies, remote arrives); every path of both CTAs
  // reaches this point, since every other wait is bounded
  if (paired) cluster_sync_all();
  if (threadIdx.x == 0) mark(SV_TRACE_EXIT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Merge split partials: O = sum_s w_s O_s / sum_s w_s, w_s = 2^(lse_s - max).
// One warp per output row.  The log2-sum-exps (lane s holds split s and
// s + 32) and the partial rows of up to 16 splits are all requested before
// any is used, so a row costs one round trip to L2 per 16 splits; empty
// splits (weight 0) may hold stale rows, so they are excluded by selection,
// never by multiplication.  It is launched as a programmatic dependent of the
// attention grid (whose CTAs signal once their partials are written) and lets
// the next grid in the stream launch early in turn.
template <int D>
__global__ void __launch_bounds__(256) split_combine_kernel(const __nv_bfloat16* __restrict__ part_o,
                                                            const float* __restrict__ part_lse,
                                                            __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                                            int rows, int splits) {
  constexpr int E = D / 32;  // elements per lane
  constexpr int kChunk = 16;
  griddep_launch_dependents();
  griddep_wait();
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float l0 = (lane < splits) ? __ldcg(part_lse + static_cast<size_t>(lane) * rows + row) : -INFINITY;
  const float l1 = (lane + 32 < splits) ? __ldcg(part_lse + static_cast<size_t>(lane + 32) * rows + row) : -INFINITY;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float mx = -INFINITY, w0 = 0.f, w1 = 0.f, wsum = 0.f;
  for (int s0 = 0; s0 < splits; s0 += kChunk) {
    uint32_t v[kChunk][E / 2];
#pragma unroll
    for (int k = 0; k < kChunk; ++k) {
#pragma unroll
      for (int e = 0; e < E / 2; ++e) v[k][e] = 0u;
      if (s0 + k < splits) {
        const __nv_bfloat16* src = part_o + (static_cast<size_t>(s0 + k) * rows + row) * D + lane * E;
        if constexpr (E == 4) {
          const uint2 t = __ldcg(reinterpret_cast<const uint2*>(src));
          v[k][0] = t.x;
          v[k][1] = t.y;
        } else {
          v[k][0] = __ldcg(reinterpret_cast<const unsigned int*>(src));
        }
      }
    }
    if (s0 == 0) {  // the weights, while the first partial rows are in flight
      mx = fmaxf(l0, l1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      w0 = (l0 == -INFINITY) ? 0.f : ex2(l0 - mx);
      w1 = (l1 == -INFINITY) ? 0.f : ex2(l1 - mx);
      wsum = w0 + w1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    }
#pragma unroll
    for (int k = 0; k < kChunk; ++k) {
      const int s = s0 + k;
      const float ws = __shfl_sync(0xffffffffu, (s < 32) ? w0 : w1, s & 31);
      if (s < splits && ws != 0.f) {
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
          acc[2 * e] += ws * __uint_as_float(v[k][e] << 16);
          acc[2 * e + 1] += ws * __uint_as_float(v[k][e] & 0xFFFF0000u);
        }
      }
    }
  }
  const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
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
  int row_tiles;
  int paired;
  int wide;  // 1: the 256-row kernel (tree_attention_wide.cu), 2: the dealt one (tree_attention_dealt.cu)
  int splits;
  int mode;
  int ctas;  // dealt kernel: resident CTAs
  size_t workspace;
};

sv_status validate(const sv_attn_params* p) {
  if (p == nullptr) return SV_ERR_INVALID_ARG;
  if (p->batch < 1 || p->num_q_heads < 1 || p->num_kv_heads < 1 || p->total_nodes < 0 || p->max_nodes < 1 ||
      p->max_pages_per_seq < 1 || p->num_pages < 1 || p->num_splits < 0 || p->max_kv_pages < 0 ||
      (p->split_reduce != 0 && p->split_reduce != 2) ||
      (p->flags & ~static_cast<int>(SV_ATTN_EARLY_CONTEXT | SV_ATTN_KERNEL_PAIRED | SV_ATTN_KERNEL_WIDE |
                                     SV_ATTN_KERNEL_DEALT)) != 0)
    return SV_ERR_INVALID_ARG;
  {
    const int k = p->flags & (SV_ATTN_KERNEL_PAIRED | SV_ATTN_KERNEL_WIDE | SV_ATTN_KERNEL_DEALT);
    if ((k & (k - 1)) != 0) return SV_ERR_INVALID_ARG;  // at most one kernel forced
  }
  if (p->num_q_heads % p->num_kv_heads != 0) return SV_ERR_INVALID_ARG;
  const int G = p->num_q_heads / p->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return SV_ERR_UNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 128) return SV_ERR_UNSUPPORTED;
  if (p->page_size != 16) return SV_ERR_UNSUPPORTED;
  if (p->max_nodes > kMaxNodes) return SV_ERR_UNSUPPORTED;
  if (p->num_splits > kMaxSplits) return SV_ERR_UNSUPPORTED;
  if (!p->q || !p->tree_k || !p->tree_v || !p->k_cache || !p->v_cache || !p->block_table || !p->ctx_lens ||
      !p->cu_nodes || !p->parents || !p->out)
    return SV_ERR_INVALID_ARG;
  if ((p->kv_pages == nullptr) != (p->cu_kv_pages == nullptr)) return SV_ERR_INVALID_ARG;
  if (!aligned16(p->q) || !aligned16(p->tree_k) || !aligned16(p->tree_v) || !aligned16(p->k_cache) ||
      !aligned16(p->v_cache) || !aligned16(p->out))
    return SV_ERR_INVALID_ARG;
  const long long row_tiles = (static_cast<long long>(p->max_nodes) * G + kTileRows - 1) / kTileRows;
  if (static_cast<long long>(p->num_kv_heads) * (row_tiles + 1) > 65535 || p->batch > 65535)
    return SV_ERR_UNSUPPORTED;
  return SV_OK;
}

template <int D>
void launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attrs, dim3 grid, bool paired, cudaStream_t s) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = grid;
  cfg->blockDim = dim3(kThreads, 1, 1);
  cfg->dynamicSmemBytes = Cfg<D>::kSmemBytes;
  cfg->stream = s;
  int n = 0;
  attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (paired) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = 1;
    attrs[n].val.clusterDim.y = 2;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg->attrs = attrs;
  cfg->numAttrs = n;
}

// One-time per-device kernel attribute (dynamic shared memory size).
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
  if (dev < 64) done[dev] = true;
  return true;
}

// Co-resident CTA pairs at this kernel's footprint (cached per device; a pair
// needs two SMs of one GPC); 0 when the query fails.
template <int D>
int max_active_pairs() {
  static std::mutex mu;
  static int cache[64];
  static bool init = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (int& v : cache) v = -1;
    init = true;
  }
  if (cache[dev] >= 0) return cache[dev];
  int n = 0;
  if (configure_kernel<D>()) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attrs[2];
    launch_config<D>(&cfg, attrs, dim3(1, 2, 1), true, nullptr);
    if (cudaOccupancyMaxActiveClusters(&n, tree_attention_kernel<D>, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cache[dev] = n;
  return n;
}

// Kernel and split count from a small cost model, in microseconds measured
// on GB300: a CTA costs a fixed prologue, first-load and epilogue time plus
// its share of K/V tiles (128 keys); waves come from how many CTAs are
// co-resident (one per SM; pairs within a GPC); splitting adds the combine
// kernel.  The paired kernel streams a tile per 128 rows in ~1.25 us, the
// 256-row kernel per 256 rows in ~2.1 us, with fixed costs of ~6.5 and
// ~8.5 us.
struct KernelCost {
  double fixed, per_tile;
  int slots;  // co-resident CTAs
  long long units;  // CTAs per split
};

double plan_cost(const KernelCost& k, int tiles, int s) {
  const long long ctas = k.units * s;
  const long long waves = (ctas + k.slots - 1) / k.slots;
  double c = static_cast<double>(waves) * (k.fixed + k.per_tile * ((tiles + s - 1) / s));
  if (s > 1) c += 5.0 + 0.05 * s;
  return c;
}

int best_splits(const KernelCost& k, int tiles, int fixed_splits, double* cost) {
  if (fixed_splits > 0) {
    *cost = plan_cost(k, tiles, fixed_splits);
    return fixed_splits;
  }
  int best_s = 1;
  double best = plan_cost(k, tiles, 1);
  for (int s = 2; s <= kMaxSplits && s <= tiles; ++s) {
    const double c = plan_cost(k, tiles, s);
    if (c < best - 1e-9) {
      best = c;
      best_s = s;
    }
  }
  *cost = best;
  return best_s;
}

// (sequence, KV head, 256-row group) slots of the dealt kernel's counters.
long long dealt_units(const sv_attn_params* p, int group) {
  return static_cast<long long>(p->batch) * p->num_kv_heads * ((static_cast<long long>(p->max_nodes) * group + 255) / 256);
}

sv_status make_plan(const sv_attn_params* p, Plan* plan) {
  sv_status st = validate(p);
  if (st != SV_OK) return st;
  plan->group = p->num_q_heads / p->num_kv_heads;
  const int rt = (p->max_nodes * plan->group + kTileRows - 1) / kTileRows;
  plan->paired = rt >= 2 ? 1 : 0;
  plan->row_tiles = plan->paired ? (rt + 1) / 2 * 2 : rt;
  const int pages = p->kv_pages ? p->max_kv_pages : p->max_pages_per_seq;
  const int tiles = (pages + kPagesPerTile - 1) / kPagesPerTile + 1;
  const bool force_paired = (p->flags & SV_ATTN_KERNEL_PAIRED) != 0;
  const bool force_wide = (p->flags & SV_ATTN_KERNEL_WIDE) != 0;
  const bool force_dealt = (p->flags & SV_ATTN_KERNEL_DEALT) != 0;
  // With an explicit split count the workspace does not depend on the
  // device, so host-only queries fall back to GB300's figures.
  int sms = 152, pairs = 76;
  if (p->num_splits == 0 || (!force_paired && !force_wide) || force_dealt) {
    const int n = device_sm_count();
    if (n > 0) {
      sms = n;
      pairs = plan->paired ? (p->head_dim == 128 ? max_active_pairs<128>() : max_active_pairs<64>()) : 0;
    } else if (p->num_splits == 0) {
      return SV_ERR_CUDA;
    }
  }
  KernelCost kp{6.5, 1.25, plan->paired && pairs > 0 ? 2 * pairs : sms,
                static_cast<long long>(p->batch) * p->num_kv_heads * plan->row_tiles};
  KernelCost kw{8.5, 2.1, sms,
                static_cast<long long>(p->batch) * p->num_kv_heads * ((p->max_nodes * plan->group + 255) / 256)};
  double cost_p = 0, cost_w = 0;
  const int sp = best_splits(kp, tiles, p->num_splits, &cost_p);
  const int sw = best_splits(kw, tiles, p->num_splits, &cost_w);
  // The dealt kernel: one CTA per SM shares the call's tiles evenly; its
  // per-tile cost is the 256-row kernel's, plus merges of the units its
  // ranges cut.  The tile count is bounded with the host's maxima.
  // a multiple of Hkv (groups of one CTA per KV head), at most 256 (a merge
  // lists at most two pieces per softmax thread)
  plan->ctas = (min(sms, 256) / p->num_kv_heads) * p->num_kv_heads;
  if (force_dealt && plan->ctas < p->num_kv_heads) return SV_ERR_UNSUPPORTED;
  const long long m_tiles = (static_cast<long long>(p->max_nodes) * plan->group + kTileRows - 1) / kTileRows;
  const long long w_est = static_cast<long long>(p->batch) * p->num_kv_heads * tiles * ((m_tiles + 1) / 2);
  const double cost_d = kw.fixed + kw.per_tile * static_cast<double>((w_est + sms - 1) / sms) + 5.0;
  // The dealt kernel is chosen only when forced: measured on GB300 its unit
  // switches cost more than the second wave they remove (serving mix 104 vs
  // 69 us for the 256-row kernel), so the model keeps the split kernels.
  (void)cost_d;
  if (force_dealt) plan->wide = 2;
  else if (force_wide) plan->wide = 1;
  else if (force_paired) plan->wide = 0;
  else plan->wide = cost_w < cost_p ? 1 : 0;
  plan->splits = plan->wide == 1 ? sw : plan->wide == 0 ? sp : 1;
  plan->mode = (plan->wide != 2 && plan->splits > 1) ? kReduceGlobal : kReduceNone;
  size_t ws = kWorkspaceHeader;
  if (plan->wide == 2) ws += dealt_workspace_bytes(plan->ctas, p->head_dim, dealt_units(p, plan->group));
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
  const cuuint64_t Hkv = p->num_kv_heads, Dd = D, P = p->page_size;
  CUtensorMap tm_kc, tm_vc, tm_tk, tm_tv;
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
  kp.q = static_cast<const __nv_bfloat16*>(p->q);
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
  kp.max_nodes = p->max_nodes;
  kp.num_splits = plan.splits;
  kp.reduce_mode = plan.mode;
  kp.early_ctx = (p->flags & SV_ATTN_EARLY_CONTEXT) ? 1 : 0;
  // measured on GB300: the tiny layer's 12 CTAs 8.22 -> 7.93 us with the
  // combine launched at once; the Llama layer's 144 CTAs slower (13.9 -> 14.8)
  kp.early_trigger = (static_cast<long long>(plan.splits) * p->num_kv_heads * plan.row_tiles * p->batch <= 32) ? 1 : 0;
  kp.total_nodes = p->total_nodes;
  kp.row_tiles = plan.row_tiles;
  kp.paired = plan.paired;
  const float scale = (p->sm_scale > 0.f) ? p->sm_scale : 1.0f / sqrtf(static_cast<float>(D));
  kp.scale_log2 = scale * 1.4426950408889634f;

  if (plan.wide == 2) {
    const size_t prow = static_cast<size_t>(plan.ctas) * 2 * 256;
    uint8_t* part = ws + kWorkspaceHeader;
    uint8_t* plse = part + align_up(prow * D * 2, 256);
    uint8_t* cnt = plse + align_up(prow * sizeof(float), 256);
    const DealtLaunch dl{plan.ctas, part, reinterpret_cast<float*>(plse), reinterpret_cast<int*>(cnt), kp.err,
                         kp.trace, kp.trace_ctas};
    return launch_dealt_attention(p, dl, stream);
  }
  if (plan.wide) {
    const WideLaunch w{plan.splits, kp.part_o, kp.part_lse, kp.err, kp.trace, kp.trace_ctas};
    const sv_status ws = launch_wide_attention(p, w, stream);
    if (ws != SV_OK) return ws;
  } else {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attrs[2];
    launch_config<D>(&cfg, attrs, dim3(plan.splits, p->num_kv_heads * plan.row_tiles, p->batch),
                     plan.paired != 0, stream);
    if (cudaLaunchKernelEx(&cfg, tree_attention_kernel<D>, tm_kc, tm_vc, tm_tk, tm_tv, kp) != cudaSuccess)
      return SV_ERR_CUDA;
  }
  if (plan.mode == kReduceGlobal) {
    cudaLaunchConfig_t ccfg = cudaLaunchConfig_t{};
    ccfg.gridDim = dim3(static_cast<unsigned>((rows * 32 + 255) / 256), 1, 1);
    ccfg.blockDim = dim3(256, 1, 1);
    ccfg.stream = stream;
    cudaLaunchAttribute cattr[1];
    cattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    cattr[0].val.programmaticStreamSerializationAllowed = 1;
    ccfg.attrs = cattr;
    ccfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&ccfg, split_combine_kernel<D>, static_cast<const __nv_bfloat16*>(kp.part_o),
                           static_cast<const float*>(kp.part_lse), kp.out, p->lse, static_cast<int>(rows),
                           plan.splits) != cudaSuccess)
      return SV_ERR_CUDA;
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

sv_status sv_tree_attention_plan(const sv_attn_params* params, int* num_splits, int* split_reduce, int* kernel) {
  if (num_splits == nullptr || split_reduce == nullptr) return SV_ERR_INVALID_ARG;
  sv::attn::Plan plan;
  const sv_status st = sv::attn::make_plan(params, &plan);
  if (st != SV_OK) return st;
  *num_splits = plan.splits;
  *split_reduce = plan.mode;
  if (kernel != nullptr) *kernel = plan.wide;
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
