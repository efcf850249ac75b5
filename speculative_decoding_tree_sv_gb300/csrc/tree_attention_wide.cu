// Tree-verification attention for sm_103a: the 256-row kernel.
//
// Same computation as the paired kernel in tree_attention.cu (SpecBlock
// Appendix A.5 and A.2; SpecPV section 3.2): out[i,h] = softmax(scale *
// q[i,h] K^T + mask) V over the context keys and the tree's
// ancestors-or-self.  Different trade-off: one CTA per (KV split, KV head x
// 256-row group, sequence) holds both 128-row tiles of a group, so every
// K/V tile is staged in exactly one SM's shared memory.  That keeps the most
// distinct bytes in flight per SM, which is what long and batched contexts
// need; short contexts that must be split many ways go to the paired kernel.
//
//   * Rows r = node * G + g; two 128-row M tiles per CTA, Q of both in shared
//     memory; K/V pages (16 tokens, head-major inside a page) gathered by TMA,
//     eight pages per 128-key tile, 128-byte swizzled, into three K and two V
//     stages (D = 128) or five of each (D = 64); the tree's K/V are one extra
//     tile.
//   * tcgen05.mma: S = Q K^T into TMEM (S0, S1), P written back as bf16 into
//     the S columns, O += P V (O0, O1) — the 512 TMEM columns.  MMA order
//     S0 S1 | PV0 S0' | PV1 S1' ... so the two softmax groups alternate.
//   * Warp roles: warp 0 loads Q and the K tiles, warp 3 the V tiles (TMA),
//     warp 1 runs the MMA schedule (converged; one elected lane issues each
//     MMA and commit), warps 4-7 and 8-11 run the softmax of the two row
//     tiles; setmaxnreg moves registers to the softmax groups.
//   * KV splits write partials (O / l in bf16 and log2-sum-exp) that the
//     combine kernel of tree_attention.cu merges.
#include <math.h>

#include <mutex>

#include "sv_device.cuh"

namespace sv {
namespace attn_wide {

constexpr int kThreads = 384;
// Registers per thread after the split: 128 x 56 (load + MMA group) + 256 x
// 224 (softmax groups) = 64512 = 384 x 168, the launch allocation.
constexpr int kRegsControl = 56;
constexpr int kRegsSoftmax = 224;
constexpr int kBlockN = 128;       // keys per tile (8 pages)
constexpr int kTileRows = 128;     // rows per M tile
constexpr int kCtaRows = 256;      // two M tiles per CTA
constexpr int kPagesPerTile = kBlockN / 16;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: defer O rescale until max grows by 2^8
constexpr float kLn2 = 0.69314718055994530942f;

enum ReduceMode : int { kReduceNone = 0, kReduceGlobal = 2 };

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;                   // 128-byte column halves
  // K stages return to the loader once their QK^T is done, V stages only
  // after PV: K may run a stage further ahead
  static constexpr int kKStages = (D == 128) ? 3 : 5;
  static constexpr int kVStages = (D == 128) ? 2 : 5;
  static constexpr uint32_t kHalfBytes = 128u * 128u;      // 128 rows x 128 B
  static constexpr uint32_t kQTileBytes = kTileRows * D * 2;
  static constexpr uint32_t kKVTileBytes = kBlockN * D * 2;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + 2 * kQTileBytes;
  static constexpr uint32_t kOffV = kOffK + kKStages * kKVTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kVStages * kKVTileBytes;
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
  static_assert(kOffBar + kBarBytes + 1024 <= 232448, "shared memory per CTA");
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
  constexpr int NSK = C::kKStages;
  constexpr int NSV = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int split = blockIdx.x;
  const int kh = blockIdx.y / p.groups_per_seq;
  const int mg = blockIdx.y % p.groups_per_seq;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
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
  uint64_t* v_full = k_full + NSK;
  uint64_t* k_empty = v_full + NSV;
  uint64_t* v_empty = k_empty + NSK;
  uint64_t* s_full = v_empty + NSV;  // [2]
  uint64_t* p_full = s_full + 2;     // [2]
  uint64_t* o_final = p_full + 2;    // [2]
  uint64_t* drain = o_final + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never_set = abort_flag + 1;  // drains wait on copies even after an abort

  // ---- prologue that reads no input: it may overlap the previous grid
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NSK; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, 1);
    }
    for (int i = 0; i < NSV; ++i) {
      mbar_init(v_full + i, 1);
      mbar_init(v_empty + i, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full + t, 1);
      mbar_init(p_full + t, kTileRows);
      mbar_init(o_final + t, 1);
    }
    mbar_init(drain, 1);
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
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) mark(SV_TRACE_PROLOGUE);
  griddep_wait();
  // without splits the next grid is the next attention call; with splits it
  // is the combine kernel, signalled once the partials are written (at exit)
  if (p.reduce_mode == kReduceNone) griddep_launch_dependents();
  if (threadIdx.x == 0) mark(SV_TRACE_INPUTS);

  // the z-th longest sequence (batches of up to 64; the index itself beyond)
  const int b = longest_first_seq(blockIdx.z, gridDim.z, p.ctx_lens, p.cu_kv_pages);
  const int n0 = p.cu_nodes[b];
  const int N = p.cu_nodes[b + 1] - n0;
  const int L = p.ctx_lens[b];
  const int rows_total = N * G;
  const int row0 = mg * kCtaRows;
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
    if (work && (warp == 0 || warp == 3)) {
      // ------------------------------------------------------------ loaders
      // warp 0 loads Q and the K tiles, warp 3 the V tiles, each as far ahead
      // as its ring allows (both resolve the tiles' page ids)
      const bool is_k = warp == 0;
      const int NS = is_k ? NSK : NSV;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* ring = smem + (is_k ? C::kOffK : C::kOffV);
      const CUtensorMap* tm_cache = is_k ? &tm_kc : &tm_vc;
      const CUtensorMap* tm_tree = is_k ? &tm_tk : &tm_tv;
      int issued = 0;
      bool ok = true;
      if (is_k && lane == 0) {
        mbar_arrive_expect_tx(q_full, (tile1 ? 2u : 1u) * C::kQTileBytes);
        for (int t = 0; t < (tile1 ? 2 : 1); ++t)
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_3d(smem + C::kOffQ + t * C::kQTileBytes + h * C::kHalfBytes, &tm_q, q_full, h * 64, kh * G,
                        n0 + (row0 + t * kTileRows) / G);
      }
      for (int it = 0; it < ntiles; ++it) {
        const int j = jb + it;
        const int st = it % NS;
        const uint32_t ph = (it / NS) & 1;
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
        if (it >= NS) {
          int w = (lane == 0) ? (mbar_wait(empty + st, ph ^ 1u, abort_flag) ? 1 : 0) : 0;
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
        }
        if (lane == 0) mbar_arrive_expect_tx(full + st, C::kKVTileBytes);
        __syncwarp();
        uint8_t* dst = ring + st * C::kKVTileBytes;
        if (ctx) {
          if (lane < kPagesPerTile)
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_4d(dst + h * C::kHalfBytes + lane * 2048, tm_cache, full + st, h * 64, 0, kh, phys);
        } else if (lane == 0) {
          for (int h = 0; h < C::kHalves; ++h) tma_load_3d(dst + h * C::kHalfBytes, tm_tree, full + st, h * 64, kh, n0);
        }
        issued = it + 1;
      }
      if (!ok && lane == 0) {
        // Timed out: stop the other roles, then let our copies land before exit.
        report_error(p.err, SV_DEVERR_TIMEOUT);
        *abort_flag = 1;
        if (is_k) mbar_wait(q_full, 0, never_set);
        for (int it = max(0, issued - NS); it < issued; ++it) mbar_wait(full + (it % NS), (it / NS) & 1, never_set);
      }
    } else if (work && warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs the schedule, so descriptors and loop state stay
      // warp-uniform; one elected lane issues each MMA and commit.  (Issuing
      // from a lane-0-only branch cost about three times the MMA's own time
      // per instruction.)
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kBlockN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
      const int nt = tile1 ? 2 : 1;
      const uint32_t q_base = smem_u32(smem + C::kOffQ);
      const uint32_t k_base = smem_u32(smem + C::kOffK);
      const uint32_t v_base = smem_u32(smem + C::kOffV);
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
      };
      auto commit = [&](uint64_t* bar) {
        if (elect_one()) umma_commit(bar);
        __syncwarp();
      };
      auto issue_qk = [&](int t, int st) {
        const uint32_t d = tmem + (t ? C::kColS1 : C::kColS0);
  #pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
          const uint64_t a = smem_desc_sw128(q_base + t * C::kQTileBytes + off, 16, 1024);
          const uint64_t bdesc = smem_desc_sw128(k_base + st * C::kKVTileBytes + off, 16, 1024);
          if (elect_one()) umma_ss(d, a, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
          __syncwarp();
        }
      };
      auto issue_pv = [&](int t, int st, bool accumulate) {
        const uint32_t d = tmem + (t ? C::kColO1 : C::kColO0);
        const uint32_t a = tmem + (t ? C::kColS1 : C::kColS0);
  #pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(v_base + st * C::kKVTileBytes + kk * 2048, C::kHalfBytes, 1024);
          if (elect_one()) umma_ts(d, a + kk * 8, bdesc, idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
          __syncwarp();
        }
      };
      bool ok = wait_all(q_full, 0);
      if (ok) ok = wait_all(k_full, 0);
      if (ok) {
        tc_fence_after();
        if (lane == 0) mark(SV_TRACE_FIRST_MMA);
        for (int t = 0; t < nt; ++t) {
          issue_qk(t, 0);
          commit(s_full + t);
        }
        commit(k_empty);
      }
      for (int it = 0; ok && it < ntiles; ++it) {
        const int vst = it % NSV;
        const uint32_t vph = (it / NSV) & 1;
        const int nx = it + 1;
        const int st2 = nx % NSK;
        const uint32_t ph2 = (nx / NSK) & 1;
        if (!wait_all(v_full + vst, vph)) { ok = false; break; }
        for (int t = 0; t < nt; ++t) {
          if (!wait_all(p_full + t, it & 1)) { ok = false; break; }
          tc_fence_after();
          issue_pv(t, vst, it > 0);
          if (nx < ntiles) {
            if (t == 0) {
              if (!wait_all(k_full + st2, ph2)) { ok = false; break; }
              tc_fence_after();
            }
            issue_qk(t, st2);
            commit(s_full + t);
          }
        }
        if (!ok) break;
        commit(v_empty + vst);
        if (nx < ntiles) commit(k_empty + st2);
      }
      if (ok) {
        for (int t = 0; t < nt; ++t) commit(o_final + t);
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
    regs_increase<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int qw = warp & 3;
    const int r = qw * 32 + lane;
    const int r_cta = t * kTileRows + r;
    const int row = row0 + r_cta;
    const bool row_exists = row < rows_total;
    const bool active = work && (t == 0 || tile1);  // warp-uniform
    // A warp whose 32 rows are all past the tree's rows only keeps the
    // barrier protocol (its S and P columns are never read back into an
    // output), which frees its scheduler's issue slots for the other warp.
    const bool warp_rows = __any_sync(0xffffffffu, row_exists);
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
          if (!warp_rows) {
            mbar_arrive(p_full + t);
            continue;
          }
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
    const bool have_o = active && ok && warp_rows;  // warp-uniform
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
      if (r_cta == 0) mark(SV_TRACE_EPILOGUE);
    } else if (p.reduce_mode == kReduceGlobal) {
      if (row_exists && (t == 0 || tile1))
        p.part_lse[static_cast<size_t>(split) * p.total_nodes * p.num_q_heads + orow] = lse2;
    }
  }
  }  // row group exists

  tc_fence_before();
  __syncthreads();
  if (p.reduce_mode != kReduceNone) griddep_launch_dependents();
  if (threadIdx.x == 0) mark(SV_TRACE_EXIT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
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

template <int D>
sv_status launch(const sv_attn_params* p, const WideLaunch& w, cudaStream_t stream) {
  if (!configure_kernel<D>()) return SV_ERR_CUDA;
  const int G = p->num_q_heads / p->num_kv_heads;
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
  Params kp;
  kp.block_table = p->block_table;
  kp.ctx_lens = p->ctx_lens;
  kp.cu_nodes = p->cu_nodes;
  kp.parents = p->parents;
  kp.kv_pages = p->kv_pages;
  kp.cu_kv_pages = p->cu_kv_pages;
  kp.out = static_cast<__nv_bfloat16*>(p->out);
  kp.lse = p->lse;
  kp.part_o = static_cast<__nv_bfloat16*>(w.part_o);
  kp.part_lse = w.part_lse;
  kp.err = w.err;
  kp.trace = w.trace;
  kp.trace_ctas = w.trace_ctas;
  kp.num_q_heads = p->num_q_heads;
  kp.group = G;
  kp.num_pages = p->num_pages;
  kp.max_pages_per_seq = p->max_pages_per_seq;
  kp.num_splits = w.splits;
  kp.reduce_mode = w.splits > 1 ? kReduceGlobal : kReduceNone;
  kp.total_nodes = p->total_nodes;
  kp.groups_per_seq = (p->max_nodes * G + kCtaRows - 1) / kCtaRows;
  const float scale = (p->sm_scale > 0.f) ? p->sm_scale : 1.0f / sqrtf(static_cast<float>(D));
  kp.scale_log2 = scale * 1.4426950408889634f;

  cudaLaunchConfig_t cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(w.splits, p->num_kv_heads * kp.groups_per_seq, p->batch);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg<D>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tree_attention_kernel<D>, tm_q, tm_kc, tm_vc, tm_tk, tm_tv, kp) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

}  // namespace attn_wide

sv_status launch_wide_attention(const sv_attn_params* p, const WideLaunch& w, cudaStream_t stream) {
  if (p->head_dim == 128) return attn_wide::launch<128>(p, w, stream);
  return attn_wide::launch<64>(p, w, stream);
}

}  // namespace sv
