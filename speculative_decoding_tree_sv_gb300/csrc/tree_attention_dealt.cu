// Tree-verification attention for sm_103a: the evenly dealt 256-row kernel.
//
// Same computation as the other two attention kernels (SpecBlock Appendix
// A.5 and A.2; SpecPV section 3.2): out[i,h] = softmax(scale * q[i,h] K^T +
// mask) V over the context keys and the tree's ancestors-or-self.  Different
// schedule: one launch of C resident CTAs (one per SM) that share the whole
// call's work evenly, whatever the batch's lengths.
//
//   * A unit is (sequence, KV head, 256-row group); its work is its context
//     tiles (128 keys each) plus the tree tile.  The CTAs form groups of Hkv,
//     one CTA per KV head: the (sequence, row group, tile) list of one head
//     is cut into equal contiguous ranges, one per group, and CTA kh of a
//     group does that range for KV head kh.  So every CTA streams the same
//     number of tiles up to one (no second wave when units outnumber the
//     SMs, no idle SMs beside long sequences), and the Hkv CTAs of a group
//     read the same pages' head slices at about the same time.
//   * A CTA walks its range unit by unit ("pieces"): the K/V ring, the MMA
//     order and every barrier phase run on across pieces, so the next piece's
//     tiles load while the previous one drains.  Q of the next piece is
//     loaded once the previous piece's last QK^T is done (q_empty); the next
//     piece's first PV overwrites O only after the softmax threads have read
//     it (their epilogue precedes their next p_full arrive).
//   * A whole unit inside a CTA writes the output; a unit cut by a range
//     boundary writes one partial per CTA piece (O / l as bf16, log2-sum-exp),
//     at most two per CTA (its first and its last piece); the piece that
//     finishes last (a counter per unit and M tile) merges them, so the call
//     is one launch.
//   * Inside a piece the engine is the 256-row kernel's: rows r = node * G +
//     g, two 128-row M tiles, Q of both in shared memory, K/V pages gathered
//     by TMA (eight 16-token pages per tile, 128-byte swizzle), tcgen05.mma
//     with S, P and O in TMEM, one producer warp, one MMA warp, two softmax
//     warpgroups; every wait is bounded.
#include <math.h>

#include <mutex>

#include "sv_device.cuh"

namespace sv {
namespace attn_dealt {

constexpr int kThreads = 384;
// Registers per thread after the split: 128 x 56 (control warps) + 256 x 224
// (softmax warpgroups) = 64512 = 384 x 168, the launch allocation.
constexpr int kRegsControl = 56;
constexpr int kRegsSoftmax = 224;
constexpr int kBlockN = 128;    // keys per tile (8 pages)
constexpr int kTileRows = 128;  // rows per M tile
constexpr int kGroupRows = 256;  // two M tiles per unit
constexpr int kPagesPerTile = kBlockN / 16;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: defer O rescale until max grows by 2^8
// The scheduler warp lists a CTA's pieces after its first in shared memory
// (the first comes straight from the range's start); a range with more
// continues with a cursor from where the list ends.
constexpr int kMaxListed = 40;
constexpr int kPieceBytes = 96;
constexpr int kCursorBytes = 112;
constexpr uint32_t kListBytes = kMaxListed * kPieceBytes + kCursorBytes + 16;
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr uint32_t kHalfBytes = 128u * 128u;
  static constexpr uint32_t kQTileBytes = kTileRows * D * 2;
  static constexpr uint32_t kKVTileBytes = kBlockN * D * 2;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + 2 * kQTileBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kKVTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kStages * kKVTileBytes;
  static constexpr uint32_t kBarBytes = 512;
  // per softmax warpgroup: the tree's parents (128 ints) and a merge's piece
  // list (256 ints); per warp of a group a piece count; the call's weight
  static constexpr uint32_t kOffPar = kOffBar + kBarBytes;   // int [2][128]
  static constexpr uint32_t kOffList = kOffPar + 2 * 128 * 4;  // int [2][256]
  static constexpr uint32_t kOffCount = kOffList + 2 * 256 * 4;  // int [2][4] + int [2] + long long
  static constexpr uint32_t kOffStage = kOffCount + 128;
  // epilogue staging: per softmax warp 8 rows of D bf16 (rows leave in four
  // passes of eight)
  static constexpr uint32_t kStageRows = 8;
  static constexpr uint32_t kStageWarpBytes = kStageRows * D * 2;
  // the CTA's pieces after its first, written by the scheduler warp
  static constexpr uint32_t kOffList2 = kOffStage + 8 * kStageWarpBytes;
  static constexpr uint32_t kSmemBytes = kOffList2 + kListBytes + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128;
  static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
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
  __nv_bfloat16* part_o;  // pieces of cut units: [C][2][256 rows][D] bf16 (O / l)
  float* part_lse;        // [C][2][256 rows] log2-sum-exp
  int* counters;          // [B * Hkv * groups_max][2] pieces finished per (unit, M tile); zero between calls
  int* err;
  unsigned long long* trace;  // optional per-CTA phase timestamps
  long long trace_ctas;
  int batch;
  int num_kv_heads;
  int num_q_heads;
  int group;  // G
  int num_pages;
  int max_pages_per_seq;
  int max_nodes;
  int groups_max;  // 256-row groups per sequence at max_nodes
  float scale_log2;
};

// What the schedule needs of sequence b.  A sequence with no node or more
// than max_nodes has no work (it is reported once, by CTA 0).
struct Seq {
  int n0, N, L, n_pages, kvp0, last_page_tokens, t_ctx, t_all, mtiles, groups;
  long long weight;  // tiles of one KV head: t_all * groups
};

__device__ __forceinline__ Seq seq_info(const Params& p, int b) {
  Seq s;
  s.n0 = p.cu_nodes[b];
  s.N = p.cu_nodes[b + 1] - s.n0;
  s.L = p.ctx_lens[b];
  s.kvp0 = 0;
  if (p.kv_pages != nullptr) {
    s.kvp0 = p.cu_kv_pages[b];
    s.n_pages = p.cu_kv_pages[b + 1] - s.kvp0;
  } else {
    s.n_pages = (max(s.L, 0) + 15) >> 4;
  }
  s.last_page_tokens = 16;
  if (s.n_pages > 0) {
    const int lp = p.kv_pages != nullptr ? p.kv_pages[s.kvp0 + s.n_pages - 1] : s.n_pages - 1;
    s.last_page_tokens = min(16, max(0, s.L - 16 * lp));
  }
  s.n_pages = max(s.n_pages, 0);
  s.t_ctx = (s.n_pages + kPagesPerTile - 1) / kPagesPerTile;
  s.t_all = s.t_ctx + 1;  // + the tree tile
  const bool valid = s.N >= 1 && s.N <= p.max_nodes;
  const int rows = valid ? s.N * p.group : 0;
  s.mtiles = (rows + kTileRows - 1) / kTileRows;
  s.groups = (rows + kGroupRows - 1) / kGroupRows;
  s.weight = static_cast<long long>(s.t_all) * s.groups;
  return s;
}

__device__ __forceinline__ long long llmin(long long a, long long b) { return a < b ? a : b; }

// Range of CTA group g of C groups: tile positions [lo, hi) of W.
__device__ __forceinline__ long long range_start(long long W, int c, int C) {
  return W * c / C;
}

// The group whose range holds tile position pos.
__device__ __forceinline__ int group_of(long long W, long long pos, int C) {
  return static_cast<int>(((pos + 1) * C - 1) / W);
}

// One unit's share of a CTA's range.
struct Piece {
  int b, kh, mg;          // the unit
  int ja, je;             // tiles [ja, je) of the unit's t_all
  int nt;                 // M tiles of the unit (1 or 2)
  int slot;               // -1: whole unit (writes the output); 0 / 1: partial slot
  long long pos;          // the unit's first tile in its head's list
  Seq s;
};

// Walks the units of one KV head that intersect [lo, hi) in order.  Every
// role of a CTA runs its own cursor over the same pieces.  Start: the first
// unit of the range (b, mg) and its first tile's position pos, as found by
// locate().
struct Cursor {
  long long lo, hi, pos;  // range, position of the current unit's first tile
  int b, kh, mg;
  Seq s;
  bool have;              // s describes sequence b
};

__device__ __forceinline__ int unit_mtiles(const Seq& s, int mg) {
  return min(2, s.mtiles - 2 * mg);
}

// Advances c to the next piece; false when the range is done.
__device__ bool next_piece(const Params& p, Cursor& c, Piece& out) {
  while (true) {
    if (c.b >= p.batch || c.pos >= c.hi) return false;
    if (!c.have) {
      c.s = seq_info(p, c.b);
      c.have = true;
    }
    if (c.s.weight == 0 || c.mg >= c.s.groups) {  // next sequence
      ++c.b;
      c.mg = 0;
      c.have = false;
      continue;
    }
    // tiles whose position lies in [lo, hi)
    const long long a = c.lo > c.pos ? c.lo - c.pos : 0;
    const long long e = c.hi - c.pos;
    const int ja = static_cast<int>(llmin(a, c.s.t_all));
    const int je = static_cast<int>(llmin(e, c.s.t_all));
    out.b = c.b;
    out.kh = c.kh;
    out.mg = c.mg;
    out.ja = ja;
    out.je = je;
    out.nt = unit_mtiles(c.s, c.mg);
    out.s = c.s;
    const bool whole = ja == 0 && je == c.s.t_all;
    out.slot = whole ? -1 : (c.pos <= c.lo ? 0 : 1);
    out.pos = c.pos;
    // advance to the next unit
    c.pos += c.s.t_all;
    if (++c.mg >= c.s.groups) {
      c.mg = 0;
      ++c.b;
      c.have = false;
    }
    if (ja < je) return true;
  }
}

// Piece k of this CTA for a role: the first from the role's own cursor, the
// next ones from the scheduler warp's list (the caller has waited for it
// before asking for piece 1), beyond the list from a cursor where the list
// ended.  False when the range is done.
__device__ bool get_piece(const Params& p, int k, Cursor& cur, Piece& pc, const Piece* list, const int* nlist,
                          const Cursor* cont) {
  if (k == 0) return next_piece(p, cur, pc);
  const int n = *nlist;
  if (k - 1 < n) {
    pc = list[k - 1];
    return true;
  }
  if (n < kMaxListed) return false;  // the list held every remaining piece
  if (k - 1 == n) cur = *cont;
  return next_piece(p, cur, pc);
}

// The unit holding position lo of group g's range (the first unit whose end
// is past lo), by one warp: per-sequence tile counts are summed in chunks of
// 32 with a warp prefix scan.  Also returns the total W.  CTA 0 reports trees
// with no node or more than max_nodes.
__device__ void locate(const Params& p, int ngroups, int g, int kh, int cta, long long* W_out, Cursor* cur) {
  const int lane = threadIdx.x & 31;
  long long tot = 0;
  for (int b0 = 0; b0 < p.batch; b0 += 32) {
    const int b = b0 + lane;
    long long w = 0;
    if (b < p.batch) {
      const Seq s = seq_info(p, b);
      w = s.weight;
      if (cta == 0 && (s.N < 1 || s.N > p.max_nodes)) report_error(p.err, SV_DEVERR_BAD_TREE);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    tot += w;
  }
  const long long W = tot;
  *W_out = W;
  cur->lo = W > 0 ? range_start(W, g, ngroups) : 0;
  cur->hi = W > 0 ? range_start(W, g + 1, ngroups) : 0;
  cur->have = false;
  cur->kh = kh;
  // sequence holding lo
  long long base = 0;
  int bsel = p.batch;
  for (int b0 = 0; b0 < p.batch && bsel == p.batch; b0 += 32) {
    const int b = b0 + lane;
    long long w = (b < p.batch) ? seq_info(p, b).weight : 0;
    long long incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, b < p.batch && base + incl > cur->lo);
    if (hit) {
      const int l = __ffs(hit) - 1;
      bsel = b0 + l;
      base += __shfl_sync(0xffffffffu, incl - w, l);
    } else {
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  cur->b = bsel;
  cur->mg = 0;
  cur->pos = base;
  if (bsel < p.batch) {
    // inside sequence b: row groups of t_all tiles each
    const Seq s = seq_info(p, bsel);
    const int mg = static_cast<int>(llmin((cur->lo - base) / s.t_all, s.groups - 1));
    cur->mg = mg;
    cur->pos = base + static_cast<long long>(s.t_all) * mg;
    cur->s = s;
    cur->have = true;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dealt_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                           const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_tk,
                           const __grid_constant__ CUtensorMap tm_tv, const __grid_constant__ Params p) {
  using C = Cfg<D>;
  constexpr int NST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int cta = blockIdx.x;
  const int ngroups = gridDim.x / p.num_kv_heads;  // the grid is a multiple of Hkv
  const int grp = cta / p.num_kv_heads;
  const int kh_cta = cta - grp * p.num_kv_heads;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* v_full = k_full + NST;
  uint64_t* k_empty = v_full + NST;
  uint64_t* v_empty = k_empty + NST;
  uint64_t* s_full = v_empty + NST;  // [2]
  uint64_t* p_full = s_full + 2;     // [2]
  uint64_t* o_final = p_full + 2;    // [2]
  uint64_t* drain = o_final + 2;
  uint64_t* list_ready = drain + 1;  // the scheduler warp has written the piece list
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(list_ready + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never_set = abort_flag + 1;
  int* par_s = reinterpret_cast<int*>(smem + C::kOffPar);
  int* list_s = reinterpret_cast<int*>(smem + C::kOffList);
  int* wcount_s = reinterpret_cast<int*>(smem + C::kOffCount);     // [2][4]
  int* flag_s = wcount_s + 8;                                       // [2]
  long long* W_s = reinterpret_cast<long long*>(smem + C::kOffCount + 48);
  Cursor* start = reinterpret_cast<Cursor*>(smem + C::kOffBar + 256);
  Piece* list = reinterpret_cast<Piece*>(smem + C::kOffList2);
  Cursor* cont = reinterpret_cast<Cursor*>(smem + C::kOffList2 + kMaxListed * kPieceBytes);
  int* nlist = reinterpret_cast<int*>(smem + C::kOffList2 + kMaxListed * kPieceBytes + kCursorBytes);
  static_assert(sizeof(Piece) <= kPieceBytes && sizeof(Cursor) <= kCursorBytes, "piece list layout");
  static_assert(256 + sizeof(Cursor) <= C::kBarBytes - 8, "schedule fits beside the barriers");
  // phase tracing (diagnostics): no live registers when it is off
  long long* trace_clk0 = reinterpret_cast<long long*>(smem + C::kOffBar + C::kBarBytes - 8);
  auto mark = [&](int ev) {
    if (p.trace != nullptr && cta < p.trace_ctas)
      p.trace[cta * kSvTraceSlots + ev] = static_cast<unsigned long long>(clock64() - *trace_clk0);
  };
  if (p.trace != nullptr && threadIdx.x == 0) {
    *trace_clk0 = clock64();
    if (cta < p.trace_ctas) p.trace[cta * kSvTraceSlots + SV_TRACE_START_NS] = globaltimer_ns();
  }

  // ---- prologue that reads no input: it may overlap the previous grid
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
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
    mbar_init(list_ready, 1);
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
  if (threadIdx.x == 0) mark(SV_TRACE_PROLOGUE);
  griddep_wait();  // the index arrays, Q and the tree's K/V may come from the preceding grid
  if (warp == 2) {
    long long W;
    Cursor cur;
    locate(p, ngroups, grp, kh_cta, cta, &W, &cur);
    if (lane == 0) {
      *start = cur;
      *W_s = W;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Cursor cur0 = *start;
  if (threadIdx.x == 0) mark(SV_TRACE_INPUTS);

  if (warp < 4) {
    regs_decrease<kRegsControl>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      Cursor cur = cur0;
      Piece pc;
      int g = 0;          // ring position over all pieces
      int k_issued = 0, v_issued = 0;
      int q_issued = 0;   // pieces whose Q was requested
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (k == 1) {
          int w = (lane == 0) ? (mbar_wait(list_ready, 0, abort_flag) ? 1 : 0) : 0;
          if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
        }
        if (!get_piece(p, k, cur, pc, list, nlist, cont)) break;
        const Seq& s = pc.s;
        const int row0 = pc.mg * kGroupRows;
        for (int j = pc.ja; j < pc.je; ++j, ++g) {
          const int st = g % NST;
          const uint32_t ph = (g / NST) & 1;
          const bool ctx = j < s.t_ctx;
          int phys = 0;
          if (ctx && lane < kPagesPerTile) {
            const int ps = min(j * kPagesPerTile + lane, s.n_pages - 1);  // ragged tail repeats the last page
            int lp = p.kv_pages != nullptr ? p.kv_pages[s.kvp0 + ps] : ps;
            if (lp < 0 || lp >= p.max_pages_per_seq) {
              report_error(p.err, SV_DEVERR_BAD_PAGE);
              lp = 0;
            }
            phys = p.block_table[static_cast<size_t>(pc.b) * p.max_pages_per_seq + lp];
            if (phys < 0 || phys >= p.num_pages) {
              report_error(p.err, SV_DEVERR_BAD_PAGE);
              phys = 0;
            }
          }
          // K tile
          if (g >= NST) {
            int w = (lane == 0) ? (mbar_wait(k_empty + st, ph ^ 1u, abort_flag) ? 1 : 0) : 0;
            if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
          }
          if (lane == 0) mbar_arrive_expect_tx(k_full + st, C::kKVTileBytes);
          __syncwarp();
          uint8_t* kdst = smem + C::kOffK + st * C::kKVTileBytes;
          if (ctx) {
            if (lane < kPagesPerTile)
              for (int h = 0; h < C::kHalves; ++h)
                tma_load_4d(kdst + h * C::kHalfBytes + lane * 2048, &tm_kc, k_full + st, h * 64, 0, pc.kh, phys);
          } else if (lane == 0) {
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_3d(kdst + h * C::kHalfBytes, &tm_tk, k_full + st, h * 64, pc.kh, s.n0);
          }
          k_issued = g + 1;
          // Q of this piece, once the previous piece's last QK^T is done (this
          // piece's first K tile is already on its way)
          if (j == pc.ja) {
            if (k > 0) {
              int w = (lane == 0) ? (mbar_wait(q_empty, (k - 1) & 1, abort_flag) ? 1 : 0) : 0;
              if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
            }
            if (lane == 0) {
              mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(pc.nt) * C::kQTileBytes);
              for (int t = 0; t < pc.nt; ++t)
                for (int h = 0; h < C::kHalves; ++h)
                  tma_load_3d(smem + C::kOffQ + t * C::kQTileBytes + h * C::kHalfBytes, &tm_q, q_full, h * 64,
                              pc.kh * G, s.n0 + (row0 + t * kTileRows) / G);
            }
            q_issued = k + 1;
            __syncwarp();
          }
          // V tile
          if (g >= NST) {
            int w = (lane == 0) ? (mbar_wait(v_empty + st, ph ^ 1u, abort_flag) ? 1 : 0) : 0;
            if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
          }
          if (lane == 0) mbar_arrive_expect_tx(v_full + st, C::kKVTileBytes);
          __syncwarp();
          uint8_t* vdst = smem + C::kOffV + st * C::kKVTileBytes;
          if (ctx) {
            if (lane < kPagesPerTile)
              for (int h = 0; h < C::kHalves; ++h)
                tma_load_4d(vdst + h * C::kHalfBytes + lane * 2048, &tm_vc, v_full + st, h * 64, 0, pc.kh, phys);
          } else if (lane == 0) {
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_3d(vdst + h * C::kHalfBytes, &tm_tv, v_full + st, h * 64, pc.kh, s.n0);
          }
          v_issued = g + 1;
        }
      }
      if (!ok && lane == 0) {
        // Timed out: stop the other roles, then let our copies land before exit.
        report_error(p.err, SV_DEVERR_TIMEOUT);
        *abort_flag = 1;
        if (q_issued > 0) mbar_wait(q_full, (q_issued - 1) & 1, never_set);
        for (int i = max(0, k_issued - NST); i < k_issued; ++i)
          mbar_wait(k_full + (i % NST), (i / NST) & 1, never_set);
        for (int i = max(0, v_issued - NST); i < v_issued; ++i)
          mbar_wait(v_full + (i % NST), (i / NST) & 1, never_set);
      }
    } else if (warp == 2) {
      // ------------------------------------------------------------ scheduler
      // Lists the CTA's pieces after the first while the first one runs, so
      // the other roles find the next unit's facts in shared memory.
      if (lane == 0) {
        Cursor c = cur0;
        Piece tmp;
        int n = 0;
        if (next_piece(p, c, tmp)) {  // the first piece: every role derives it itself
          while (n < kMaxListed && next_piece(p, c, tmp)) list[n++] = tmp;
        }
        *cont = c;
        *nlist = n;
        mbar_arrive(list_ready);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs the schedule (warp-uniform descriptors and loop
      // state); one elected lane issues each MMA and commit.
      {
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
          return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
        };
        auto commit = [&](uint64_t* bar) {
          if (elect_one()) umma_commit(bar);
          __syncwarp();
        };
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kBlockN, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
        const uint32_t q_base = smem_u32(smem + C::kOffQ);
        const uint32_t k_base = smem_u32(smem + C::kOffK);
        const uint32_t v_base = smem_u32(smem + C::kOffV);
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
        Cursor cur = cur0;
        Piece pc;
        bool ok = true;
        int g = 0;                // ring position of the piece's first tile
        int tiles_t[2] = {0, 0};  // tiles handed to each M tile's softmax before this piece
        for (int k = 0; ok; ++k) {
          if (k == 1 && !wait_all(list_ready, 0)) { ok = false; break; }
          if (!get_piece(p, k, cur, pc, list, nlist, cont)) break;
          const int nt = pc.nt;
          const int n = pc.je - pc.ja;
          const int st0 = g % NST;
          ok = wait_all(q_full, k & 1) && wait_all(k_full + st0, (g / NST) & 1);
          if (!ok) break;
          tc_fence_after();
          if (k == 0 && lane == 0) mark(SV_TRACE_FIRST_MMA);
          for (int t = 0; t < nt; ++t) {
            issue_qk(t, st0);
            commit(s_full + t);
          }
          commit(k_empty + st0);
          if (n == 1) commit(q_empty);  // the piece's last QK^T is issued
          for (int it = 0; ok && it < n; ++it) {
            const int gg = g + it;
            const int st = gg % NST;
            const uint32_t ph = (gg / NST) & 1;
            const int nx = it + 1;
            const int st2 = (gg + 1) % NST;
            const uint32_t ph2 = ((gg + 1) / NST) & 1;
            if (!wait_all(v_full + st, ph)) { ok = false; break; }
            for (int t = 0; t < nt; ++t) {
              if (!wait_all(p_full + t, (tiles_t[t] + it) & 1)) { ok = false; break; }
              tc_fence_after();
              issue_pv(t, st, it > 0);
              if (nx < n) {
                if (t == 0) {
                  if (!wait_all(k_full + st2, ph2)) { ok = false; break; }
                  tc_fence_after();
                }
                issue_qk(t, st2);
                commit(s_full + t);
              }
            }
            if (!ok) break;
            commit(v_empty + st);
            if (nx < n) {
              commit(k_empty + st2);
              if (nx == n - 1) commit(q_empty);
            }
          }
          if (!ok) break;
          for (int t = 0; t < nt; ++t) commit(o_final + t);
          g += n;
          for (int t = 0; t < nt; ++t) tiles_t[t] += n;
        }
        if (!ok) {
          if (lane == 0) {
            report_error(p.err, SV_DEVERR_TIMEOUT);
            *abort_flag = 1;
          }
          commit(drain);  // let issued MMAs finish before TMEM is freed
          __all_sync(0xffffffffu, mbar_wait(drain, 0, never_set));
        }
      }
      __syncwarp();
    }
  } else {
    regs_increase<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;  // M tile
    const int qw = warp & 3;
    const int r = qw * 32 + lane;   // TMEM lane = row of the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    const uint32_t col_s = t ? C::kColS1 : C::kColS0;
    const uint32_t col_o = t ? C::kColO1 : C::kColO0;
    int* par_t = par_s + t * 128;
    int* list_t = list_s + t * 256;
    uint8_t* stage = smem + C::kOffStage + (warp - 4) * C::kStageWarpBytes;
    int tiles_done = 0, pieces_done = 0;
    bool ok = true;
    Cursor cur = cur0;
    Piece pc;
    Piece cut[2];  // this CTA's pieces of cut units (its first and its last), merged at the end
    int ncut = 0;
    for (int k = 0; ok; ++k) {
      if (k == 1 && !__all_sync(0xffffffffu, mbar_wait(list_ready, 0, abort_flag))) { ok = false; break; }
      if (!get_piece(p, k, cur, pc, list, nlist, cont)) break;
      if (t >= pc.nt) continue;  // this M tile has no rows in the unit
      const Seq& s = pc.s;
      const int row = pc.mg * kGroupRows + t * kTileRows + r;
      const int rows_total = s.N * G;
      const bool row_exists = row < rows_total;
      const int node = row / G;
      const int gq = row - node * G;
      // The tree's parents are requested now (one per thread: N <= 128) and
      // staged in shared memory at the tree tile, where each row walks its
      // ancestor chain there: no dependent global load on the way.
      const bool has_tree = pc.je == s.t_all;
      int my_par = -1;
      if (has_tree && r < s.N) my_par = p.parents[s.n0 + r];
      uint32_t anc0 = 0, anc1 = 0, anc2 = 0, anc3 = 0;
      float m_run = -INFINITY;
      float l_run = 0.f;
      const int n = pc.je - pc.ja;
      for (int it = 0; it < n; ++it) {
        const int j = pc.ja + it;
        if (j >= s.t_ctx) {
          // the tree tile (the piece's last): every row's ancestor-or-self set
          par_t[r] = my_par;
          named_barrier(2 + t, kTileRows);
          if (row_exists) {
            int c = node;
            for (int step = 0; step < kMaxNodes && c >= 0 && c < kMaxNodes; ++step) {
              const uint32_t bit = 1u << (c & 31);
              if ((c >> 5) == 0) anc0 |= bit;
              else if ((c >> 5) == 1) anc1 |= bit;
              else if ((c >> 5) == 2) anc2 |= bit;
              else anc3 |= bit;
              if (c == 0) break;
              const int pcn = par_t[c];
              if (pcn < 0 || pcn >= c) {
                report_error(p.err, SV_DEVERR_BAD_PARENT);
                break;
              }
              c = pcn;
            }
          }
        }
        // warp-uniform outcome: the TMEM loads below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(s_full + t, (tiles_done + it) & 1, abort_flag))) { ok = false; break; }
        tc_fence_after();
        if (tiles_done + it == 0 && t == 0 && r == 0) mark(SV_TRACE_FIRST_S);
        uint32_t sr[kBlockN];
#pragma unroll
        for (int c = 0; c < kBlockN / 32; ++c)
          tmem_ld32(lane_base + col_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + c * 32));
        tmem_ld_wait();
        // mask: only the ragged last context tile and the tree tile need one
        constexpr uint32_t kNegInf = 0xFF800000u;
        if (j >= s.t_ctx) {
#pragma unroll
          for (int kk = 0; kk < kBlockN; ++kk) {
            const uint32_t w = (kk < 32) ? anc0 : (kk < 64) ? anc1 : (kk < 96) ? anc2 : anc3;
            if (!((kk < s.N) && ((w >> (kk & 31)) & 1u))) sr[kk] = kNegInf;
          }
        } else if (j == s.t_ctx - 1) {
          const int nvalid = (s.n_pages - kPagesPerTile * j - 1) * 16 + s.last_page_tokens;
#pragma unroll
          for (int kk = 0; kk < kBlockN; ++kk)
            if (kk >= nvalid) sr[kk] = kNegInf;
        }
        // row maximum of the raw scores (scale > 0 commutes with max)
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int kk = 0; kk < kBlockN; kk += 8) {
          mx0 = max3(mx0, __uint_as_float(sr[kk + 0]), __uint_as_float(sr[kk + 1]));
          mx1 = max3(mx1, __uint_as_float(sr[kk + 2]), __uint_as_float(sr[kk + 3]));
          mx2 = max3(mx2, __uint_as_float(sr[kk + 4]), __uint_as_float(sr[kk + 5]));
          mx3 = max3(mx3, __uint_as_float(sr[kk + 6]), __uint_as_float(sr[kk + 7]));
        }
        const float tmax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * p.scale_log2;
        const float m_new = fmaxf(m_run, tmax);
        const bool grow = m_new > m_run + kRescaleThreshold;
        // O holds the piece's earlier tiles (their PV finished before this S
        // was committed): rescale it and the running sum, the whole warp
        // together (warp-collective TMEM access; rows that need none scale
        // by 1)
        if (it > 0 && __any_sync(0xffffffffu, grow)) {
          const float f = grow ? ex2(m_run - m_new) : 1.f;
          l_run *= f;
          const uint64_t f2 = f2_pack(f, f);
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            tmem_ld32(lane_base + col_o + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int kk = 0; kk < 32; kk += 2) {
              const uint64_t v = f2_mul(f2_pack(__uint_as_float(o[kk]), __uint_as_float(o[kk + 1])), f2);
              o[kk] = static_cast<uint32_t>(v);
              o[kk + 1] = static_cast<uint32_t>(v >> 32);
            }
            tmem_st32(lane_base + col_o + c * 32, o);
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
        for (int kk = 0; kk < kBlockN; kk += 4) {
          const uint64_t a = f2_fma(f2_pack(__uint_as_float(sr[kk]), __uint_as_float(sr[kk + 1])), sc2, nm2);
          const uint64_t b2 = f2_fma(f2_pack(__uint_as_float(sr[kk + 2]), __uint_as_float(sr[kk + 3])), sc2, nm2);
          const float p0 = ex2(f2_lo(a)), p1 = ex2(f2_hi(a));
          const float p2 = ex2(f2_lo(b2)), p3 = ex2(f2_hi(b2));
          acc0 = f2_add(acc0, f2_pack(p0, p1));
          acc1 = f2_add(acc1, f2_pack(p2, p3));
          pk[kk >> 1] = pack_bf16x2(p0, p1);
          pk[(kk >> 1) + 1] = pack_bf16x2(p2, p3);
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
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_final + t, pieces_done & 1, abort_flag));
      if (!ok) break;
      if (t == 0 && r == 0) mark(SV_TRACE_O_READY);
      // ---------------------------------------------------------- epilogue
      // O / l of this thread's row as bf16 (the TMEM loads complete before the
      // next piece's first P is handed over, which is what lets that piece's
      // first PV overwrite O), then out through shared memory so that the
      // global stores are coalesced: the rings already hold the next piece's
      // tiles, so every warp has a staging area of its own for eight rows;
      // 16-byte chunks sit XOR-swizzled by row to keep the writes conflict-free.
      tc_fence_after();
      const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
      const size_t orow = static_cast<size_t>(s.n0 + node) * p.num_q_heads + pc.kh * G + gq;
      const int prow = t * kTileRows + r;  // row within the unit's 256-row group
      __nv_bfloat16* const dst_row =
          pc.slot < 0 ? p.out + orow * D
                      : p.part_o + ((static_cast<size_t>(cta) * 2 + pc.slot) * kGroupRows + prow) * D;
      constexpr int kChunks = D / 8;  // 16-byte chunks per row
      uint32_t ob[D / 2];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_base + col_o + c * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int k2 = 0; k2 < 16; ++k2)
          ob[c * 16 + k2] = pack_bf16x2(__uint_as_float(o[2 * k2]) * inv_l, __uint_as_float(o[2 * k2 + 1]) * inv_l);
      }
      {
        constexpr int kRowsPerStore = 32 / kChunks;       // rows one warp store covers
        constexpr int kStores = C::kStageRows / kRowsPerStore;
        const unsigned long long my_dst = reinterpret_cast<unsigned long long>(dst_row);
        const int my_ok = row_exists ? 1 : 0;
#pragma unroll
        for (int pass = 0; pass < 32 / static_cast<int>(C::kStageRows); ++pass) {
          if ((lane / C::kStageRows) == static_cast<unsigned>(pass)) {
            const int sr_ = lane % C::kStageRows;
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch) {
              const int pos = ch ^ (sr_ % kChunks);
              *reinterpret_cast<uint4*>(stage + sr_ * (D * 2) + pos * 16) =
                  make_uint4(ob[4 * ch], ob[4 * ch + 1], ob[4 * ch + 2], ob[4 * ch + 3]);
            }
          }
          __syncwarp();
#pragma unroll
          for (int k2 = 0; k2 < kStores; ++k2) {
            const int sr_ = k2 * kRowsPerStore + lane / kChunks;  // staged row
            const int src_lane = pass * C::kStageRows + sr_;
            const unsigned long long d = __shfl_sync(0xffffffffu, my_dst, src_lane);
            const int okr = __shfl_sync(0xffffffffu, my_ok, src_lane);
            const int ch = lane % kChunks;
            const uint4 v = *reinterpret_cast<const uint4*>(stage + sr_ * (D * 2) + (ch ^ (sr_ % kChunks)) * 16);
            if (okr) reinterpret_cast<uint4*>(d)[ch] = v;
          }
          __syncwarp();
        }
      }
      if (row_exists) {
        const float lse2 = (l_run > 0.f) ? m_run + log2f(l_run) : -INFINITY;
        if (pc.slot < 0) {
          if (p.lse != nullptr) p.lse[orow] = lse2 * kLn2;
        } else {
          p.part_lse[(static_cast<size_t>(cta) * 2 + pc.slot) * kGroupRows + prow] = lse2;
        }
      }
      if (pc.slot >= 0 && ncut < 2) cut[ncut++] = pc;
      tiles_done += n;
      ++pieces_done;
      if (t == 0 && r == 0) mark(SV_TRACE_EPILOGUE);
    }
    // ---------------------------------------------------- merges of cut units
    // A cut unit's pieces are in the groups first..last whose ranges hold its
    // tiles (an empty range holds none), at the CTA of the unit's KV head.  Each piece
    // counts itself once this CTA is done with its pieces; the last to count
    // merges them all (no waiting on another CTA) and leaves the counter at
    // zero for the next call.  Counting at the end keeps the count's round
    // trip off the pipeline.
    for (int ci = 0; ok && ci < ncut; ++ci) {
      const Piece& q = cut[ci];
      const Seq& s = q.s;
      const int row = q.mg * kGroupRows + t * kTileRows + r;
      const bool row_exists = row < s.N * G;
      const int node = row / G;
      const int gq = row - node * G;
      const size_t orow = static_cast<size_t>(s.n0 + node) * p.num_q_heads + q.kh * G + gq;
      const int prow = t * kTileRows + r;
      const long long W = *W_s;
      const int first = group_of(W, q.pos, ngroups);  // groups holding the unit's first and last tiles
      const int last = group_of(W, q.pos + s.t_all - 1, ngroups);
      const int span = last - first + 1;  // <= 256 (one CTA per SM)
      // the list of pieces, in CTA order: per warp of the group a ballot,
      // the warps' counts in shared memory, then each warp's base
      int total = 0;
      for (int i0 = 0; i0 < span; i0 += kTileRows) {
        const int i = i0 + r;
        bool holds = false;
        int base_row = 0;
        if (i < span) {
          const int g = first + i;
          const long long lo = range_start(W, g, ngroups), hi = range_start(W, g + 1, ngroups);
          const long long ja = lo > q.pos ? lo - q.pos : 0;
          holds = ja < s.t_all && q.pos + ja < hi;
          const int c = g * p.num_kv_heads + q.kh;  // that group's CTA for this KV head
          base_row = (c * 2 + (q.pos <= lo ? 0 : 1)) * kGroupRows;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, holds);
        if (lane == 0) wcount_s[t * 4 + qw] = __popc(bal);
        named_barrier(4 + t, kTileRows);
        int base = total;
        for (int w = 0; w < qw; ++w) base += wcount_s[t * 4 + w];
        if (holds) list_t[base + __popc(bal & ((1u << lane) - 1u))] = base_row;
        for (int w = 0; w < 4; ++w) total += wcount_s[t * 4 + w];
        named_barrier(4 + t, kTileRows);
      }
      // count this piece once every thread's partial rows are visible
      // device-wide (each fences its own writes; the barrier orders the
      // fences before thread 0's count)
      const int u = (q.b * p.num_kv_heads + q.kh) * p.groups_max + q.mg;
      __threadfence();
      named_barrier(4 + t, kTileRows);
      if (r == 0) flag_s[t] = atomicAdd(p.counters + 2 * u + t, 1) == total - 1 ? 1 : 0;
      named_barrier(4 + t, kTileRows);
      if (!flag_s[t]) continue;
      if (r == 0) p.counters[2 * u + t] = 0;
      __threadfence();
      if (!row_exists) continue;
      constexpr int kChunks = D / 8;
      uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D);
      if (total <= 2) {
        // the common case: both rows and both log2-sum-exps in one round trip
        float l2[2] = {-INFINITY, -INFINITY};
        uint4 v[2][kChunks];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (i < total) {
            const size_t pr = static_cast<size_t>(list_t[i]) + prow;
            l2[i] = __ldcg(p.part_lse + pr);
            const uint4* src = reinterpret_cast<const uint4*>(p.part_o + pr * D);
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch) v[i][ch] = __ldcg(src + ch);
          } else {
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch) v[i][ch] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        const float mx = fmaxf(l2[0], l2[1]);
        const float w0 = (l2[0] == -INFINITY) ? 0.f : ex2(l2[0] - mx);
        const float w1 = (l2[1] == -INFINITY) ? 0.f : ex2(l2[1] - mx);
        const float ws = w0 + w1;
        const float inv = (ws > 0.f) ? 1.f / ws : 0.f;
        const float a0 = w0 * inv, a1 = w1 * inv;
#pragma unroll
        for (int ch = 0; ch < kChunks; ++ch) {
          const uint32_t x0[4] = {v[0][ch].x, v[0][ch].y, v[0][ch].z, v[0][ch].w};
          const uint32_t x1[4] = {v[1][ch].x, v[1][ch].y, v[1][ch].z, v[1][ch].w};
          uint32_t o4[4];
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) {
            const float lo = a0 * __uint_as_float(x0[k2] << 16) + a1 * __uint_as_float(x1[k2] << 16);
            const float hi = a0 * __uint_as_float(x0[k2] & 0xFFFF0000u) + a1 * __uint_as_float(x1[k2] & 0xFFFF0000u);
            o4[k2] = pack_bf16x2(lo, hi);
          }
          dst[ch] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
        }
        if (p.lse != nullptr) p.lse[orow] = (ws > 0.f) ? (mx + log2f(ws)) * kLn2 : -INFINITY;
      } else {
        // more pieces (a unit longer than a CTA's share): an online merge,
        // one piece's row in flight at a time
        float acc[D];
#pragma unroll
        for (int e = 0; e < D; ++e) acc[e] = 0.f;
        float mx = -INFINITY, wsum = 0.f;
        for (int i = 0; i < total; ++i) {
          const size_t pr = static_cast<size_t>(list_t[i]) + prow;
          const float li = __ldcg(p.part_lse + pr);
          const uint4* src = reinterpret_cast<const uint4*>(p.part_o + pr * D);
          uint4 v[kChunks];
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch) v[ch] = __ldcg(src + ch);
          if (li == -INFINITY) continue;
          if (li > mx) {
            const float f = (mx == -INFINITY) ? 0.f : ex2(mx - li);
            wsum *= f;
#pragma unroll
            for (int e = 0; e < D; ++e) acc[e] *= f;
            mx = li;
          }
          const float w = ex2(li - mx);
          wsum += w;
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch) {
            const uint32_t x[4] = {v[ch].x, v[ch].y, v[ch].z, v[ch].w};
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
              acc[ch * 8 + 2 * k2] += w * __uint_as_float(x[k2] << 16);
              acc[ch * 8 + 2 * k2 + 1] += w * __uint_as_float(x[k2] & 0xFFFF0000u);
            }
          }
        }
        const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
#pragma unroll
        for (int ch = 0; ch < kChunks; ++ch)
          dst[ch] = make_uint4(pack_bf16x2(acc[ch * 8 + 0] * inv, acc[ch * 8 + 1] * inv),
                               pack_bf16x2(acc[ch * 8 + 2] * inv, acc[ch * 8 + 3] * inv),
                               pack_bf16x2(acc[ch * 8 + 4] * inv, acc[ch * 8 + 5] * inv),
                               pack_bf16x2(acc[ch * 8 + 6] * inv, acc[ch * 8 + 7] * inv));
        if (p.lse != nullptr) p.lse[orow] = (wsum > 0.f) ? (mx + log2f(wsum)) * kLn2 : -INFINITY;
      }
    }
    if (!ok && lane == 0) {
      report_error(p.err, SV_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  griddep_launch_dependents();  // the partials are written: the combine may run
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
  if (cudaFuncSetAttribute(dealt_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<D>::kSmemBytes) != cudaSuccess)
    return false;
  if (dev < 64) done[dev] = true;
  return true;
}

template <int D>
sv_status launch(const sv_attn_params* p, const DealtLaunch& w, cudaStream_t stream) {
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
  kp.counters = w.counters;
  kp.err = w.err;
  kp.trace = w.trace;
  kp.trace_ctas = w.trace_ctas;
  kp.batch = p->batch;
  kp.num_kv_heads = p->num_kv_heads;
  kp.num_q_heads = p->num_q_heads;
  kp.group = G;
  kp.num_pages = p->num_pages;
  kp.max_pages_per_seq = p->max_pages_per_seq;
  kp.max_nodes = p->max_nodes;
  kp.groups_max = (p->max_nodes * G + kGroupRows - 1) / kGroupRows;
  const float scale = (p->sm_scale > 0.f) ? p->sm_scale : 1.0f / sqrtf(static_cast<float>(D));
  kp.scale_log2 = scale * 1.4426950408889634f;

  cudaLaunchConfig_t cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(static_cast<unsigned>(w.ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg<D>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, dealt_attention_kernel<D>, tm_q, tm_kc, tm_vc, tm_tk, tm_tv, kp) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

}  // namespace attn_dealt

size_t dealt_workspace_bytes(int ctas, int head_dim, long long units) {
  const size_t rows = static_cast<size_t>(ctas) * 2 * attn_dealt::kGroupRows;
  return align_up(rows * head_dim * 2, 256) + align_up(rows * sizeof(float), 256) +
         align_up(static_cast<size_t>(units) * 2 * sizeof(int), 256);
}

sv_status launch_dealt_attention(const sv_attn_params* p, const DealtLaunch& w, cudaStream_t stream) {
  if (p->head_dim == 128) return attn_dealt::launch<128>(p, w, stream);
  return attn_dealt::launch<64>(p, w, stream);
}

}  // namespace sv
